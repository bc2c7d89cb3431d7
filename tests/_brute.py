"""Pure-Python scalar brute force of the GroupQueryAttention forward pass.

A second, independently written formulation used only to pin the numpy
oracle on tiny shapes: scalar loops over every index, rotary of queries as a
complex multiplication, their RMS norm and every sum through ``math.fsum``,
the softmax as exp(s - logsumexp) with the sink logit inside the log-sum-exp;
stored K rows through a scalar fp32 restatement of the stored-row recipe
(recursive pairwise tree). It shares no code with ``oracle/``.
"""

import math

import numpy as np


def _f(x):
    return float(x)


# Stored K rows follow the fp32 recipe: every operation rounded to fp32 (a
# double result of two fp32 operands rounds to the correctly rounded fp32
# result for +, -, *, / and sqrt), squares summed left to right in groups of
# four, the group sums added as a balanced binary tree (recursive halving of
# the group list padded with zeros to a power of two).
def f32(x):
    return float(np.float32(x))


def _tree32(vals):
    if len(vals) == 1:
        return vals[0]
    mid = len(vals) // 2
    return f32(_tree32(vals[:mid]) + _tree32(vals[mid:]))


def norm32(vec, w, eps):
    """Scalar fp32 RMS norm of one row (list of fp32 values as Python floats)."""
    groups = []
    for g0 in range(0, len(vec), 4):
        acc = f32(vec[g0] * vec[g0])
        for d in range(g0 + 1, g0 + 4):
            acc = f32(acc + f32(vec[d] * vec[d]))
        groups.append(acc)
    width = 1
    while width < len(groups):
        width *= 2
    ss = _tree32(groups + [0.0] * (width - len(groups)))
    ms = f32(ss / len(vec))
    r = f32(1.0 / f32(math.sqrt(f32(ms + f32(eps)))))
    return [f32(f32(vec[d] * r) * _f(w[d])) for d in range(len(vec))]


def rope32(vec, cos_row, sin_row):
    """Scalar fp32 NeoX rotary of one row: rounded products, then one rounded add / subtract."""
    half = len(vec) // 2
    outv = list(vec)
    for d in range(half):
        c, s_ = _f(cos_row[d]), _f(sin_row[d])
        a, b2 = vec[d], vec[d + half]
        outv[d] = f32(f32(a * c) - f32(b2 * s_))
        outv[d + half] = f32(f32(b2 * c) + f32(a * s_))
    return outv


def brute_forward(inputs, attrs, present_key, present_value, share_buffer):
    N = attrs["num_heads"]
    Nkv = attrs["kv_num_heads"]
    q = inputs["query"]
    k = inputs["key"]
    v = inputs["value"]
    B, S, hq = q.shape
    H = hq // N
    G = N // Nkv
    half = H // 2
    has_past = inputs.get("past_key") is not None
    if share_buffer:
        pk = [[[r.copy() for r in inputs["past_key"][b, g]] for g in range(Nkv)] for b in range(B)]
        pv = [[[r.copy() for r in inputs["past_value"][b, g]] for g in range(Nkv)] for b in range(B)]
        cache_dtype = inputs["past_key"].dtype
    else:
        pk = [[[r.copy() for r in present_key[b, g]] for g in range(Nkv)] for b in range(B)]
        pv = [[[r.copy() for r in present_value[b, g]] for g in range(Nkv)] for b in range(B)]
        cache_dtype = present_key.dtype
    quant = attrs.get("k_quant_type", "NONE") != "NONE"
    # prompt with a float cache of another dtype: attention reads the rows in the query dtype
    separate = not quant and not has_past and np.dtype(cache_dtype) != q.dtype
    ak = [[[None] * len(pk[b][g]) for g in range(Nkv)] for b in range(B)]
    av = [[[None] * len(pv[b][g]) for g in range(Nkv)] for b in range(B)]
    int4 = quant and attrs.get("kv_cache_bit_width", 8) == 4
    qmax = 7 if int4 else 127
    eps = attrs.get("qk_norm_epsilon", 1e-6)
    qw = inputs.get("q_norm_weight")
    kw = inputs.get("k_norm_weight")
    rotary = attrs.get("do_rotary", 0) == 1
    cosc = inputs.get("cos_cache")
    sinc = inputs.get("sin_cache")
    scale = attrs.get("scale", 0.0) or 1.0 / math.sqrt(H)
    cap = attrs.get("softcap", 0.0)
    W = attrs.get("local_window_size", -1)
    causal = attrs.get("causal", 1) == 1
    bias = inputs.get("attention_bias")
    sink = inputs.get("head_sink")
    smooth = attrs.get("smooth_softmax", -1) == 1

    def norm(vec, w):
        ms = math.fsum(x * x for x in vec) / len(vec)
        r = 1.0 / math.sqrt(ms + eps)
        return [vec[d] * r * _f(w[d]) for d in range(len(vec))]

    def rope(vec, pos):
        outv = list(vec)
        for d in range(half):
            z = complex(vec[d], vec[d + half]) * complex(_f(cosc[pos, d]), _f(sinc[pos, d]))
            outv[d], outv[d + half] = z.real, z.imag
        return outv

    def scales(name, g):
        sc = inputs[name].reshape(-1)
        return [_f(sc[0]) if sc.size == 1 else _f(sc[g * H + d]) for d in range(H)]

    def store(vec, g, name):
        if quant:
            sc = inputs[name].reshape(-1)
            codes = []
            for d in range(H):
                s32 = sc[0] if sc.size == 1 else sc[g * H + d]
                t = np.float32(vec[d]) / np.float32(s32)
                codes.append(max(-qmax, min(qmax, round(float(t)))))   # Python round: ties to even
            if int4:   # byte k = biased code of 2k + 16 * biased code of 2k+1
                return np.array([(codes[2 * k] + 8) + 16 * (codes[2 * k + 1] + 8) for k in range(H // 2)],
                                dtype=np.uint8)
            return np.array(codes, dtype=np.int8)
        return np.array(vec, dtype=np.float64).astype(cache_dtype)

    def value(row, g, name):
        if quant:
            sc = scales(name, g)
            if int4:
                codes = []
                for byte in row:
                    codes += [int(byte) % 16 - 8, int(byte) // 16 - 8]
                return [codes[d] * sc[d] for d in range(H)]
            return [int(row[d]) * sc[d] for d in range(H)]
        return [_f(x) for x in row]

    out = np.zeros((B, S, N * H))
    for b in range(B):
        total = int(inputs["seqlens_k"][b]) + 1
        past = total - S if has_past else 0
        if has_past and not share_buffer:
            for g in range(Nkv):
                for j in range(past):
                    pk[b][g][j] = inputs["past_key"][b, g, j].copy()
                    pv[b][g][j] = inputs["past_value"][b, g, j].copy()
        for g in range(Nkv):
            for i in range(S):
                kr = [_f(x) for x in k[b, i, g * H:(g + 1) * H]]   # exact: T is fp16 or fp32
                vr = [_f(x) for x in v[b, i, g * H:(g + 1) * H]]
                if kw is not None:
                    kr = norm32(kr, kw, eps)
                if rotary:
                    kr = rope32(kr, cosc[past + i], sinc[past + i])
                pk[b][g][past + i] = store(kr, g, "k_scale")
                pv[b][g][past + i] = store(vr, g, "v_scale")
                if separate:
                    ak[b][g][past + i] = np.array(kr, dtype=np.float64).astype(q.dtype)
                    av[b][g][past + i] = np.array(vr, dtype=np.float64).astype(q.dtype)
        for h in range(N):
            g = h // G
            for i in range(S):
                if not has_past and i >= total:
                    continue
                pos = past + i
                qr = [_f(x) for x in q[b, i, h * H:(h + 1) * H]]
                if qw is not None:
                    qr = norm(qr, qw)
                if rotary:
                    qr = rope(qr, pos)
                logits = []
                for j in range(total):
                    if causal and j > pos:
                        continue
                    if W >= 0 and j < pos - W:
                        continue
                    kj = value(ak[b][g][j] if separate else pk[b][g][j], g, "k_scale")
                    s = scale * math.fsum(qr[d] * kj[d] for d in range(H))
                    if cap > 0:
                        s = cap * math.tanh(s / cap)
                    if bias is not None:
                        bb = 0 if bias.shape[0] == 1 else b
                        bh = 0 if bias.shape[1] == 1 else h
                        s += _f(bias[bb, bh, i, j])
                    logits.append((j, s))
                sig = None
                if sink is not None:
                    sig = _f(sink[h])
                elif smooth:
                    sig = 0.0
                allv = [s for _, s in logits] + ([sig] if sig is not None else [])
                mx = max(allv)
                lse = mx + math.log(math.fsum(math.exp(s - mx) for s in allv))
                for d in range(H):
                    terms = []
                    for j, s in logits:
                        vj = av[b][g][j] if separate else pv[b][g][j]
                        terms.append(math.exp(s - lse) * value(vj, g, "v_scale")[d])
                    out[b, i, h * H + d] = math.fsum(terms)
    pk_arr = np.array([[np.stack(pk[b][g]) for g in range(Nkv)] for b in range(B)])
    pv_arr = np.array([[np.stack(pv[b][g]) for g in range(Nkv)] for b in range(B)])
    return out, pk_arr, pv_arr
