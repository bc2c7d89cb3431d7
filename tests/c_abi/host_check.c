/* Host-only use of the C ABI from plain C (no CUDA call is made): the header
 * compiles as C11, the library links, defaults and status strings are as
 * declared, and the host-side checks accept a valid decode call and reject a
 * broken one. Device pointers are fake 256-byte-aligned addresses (never
 * dereferenced by the host checks). Exit status 0 on success. */
#include <stdio.h>
#include <string.h>

#include "gqa.h"

static gqa_tensor t4(uintptr_t addr, int32_t dtype, int ndim, int64_t a, int64_t b, int64_t c, int64_t d) {
  gqa_tensor t;
  memset(&t, 0, sizeof(t));
  t.data = (void*)addr;
  t.dtype = dtype;
  t.ndim = ndim;
  t.shape[0] = a;
  t.shape[1] = b;
  t.shape[2] = c;
  t.shape[3] = d;
  return t;
}

int main(void) {
  gqa_attrs a;
  gqa_attrs_default(&a);
  if (a.causal != 1 || a.local_window_size != -1 || a.smooth_softmax != -1 || a.kv_cache_bit_width != 8) return 1;
  if (strcmp(gqa_status_string(GQA_ERR_UNSUPPORTED), "GQA_ERR_UNSUPPORTED") != 0) return 2;
  a.num_heads = 8;
  a.kv_num_heads = 2;
  gqa_handle* h = NULL;
  if (gqa_create(&a, &h) != GQA_OK || h == NULL) return 3;

  /* fp16 decode over a shared cache: B=2, S=1, N=8, N_kv=2, H=128, C=64. */
  gqa_inputs in;
  gqa_outputs out;
  memset(&in, 0, sizeof(in));
  memset(&out, 0, sizeof(out));
  uintptr_t next = 0x100000;
#define NEXT() (next += (uintptr_t)1 << 24)
  in.query = t4(NEXT(), GQA_F16, 3, 2, 1, 8 * 128, 0);
  in.key = t4(NEXT(), GQA_F16, 3, 2, 1, 2 * 128, 0);
  in.value = t4(NEXT(), GQA_F16, 3, 2, 1, 2 * 128, 0);
  in.seqlens_k = t4(NEXT(), GQA_I32, 1, 2, 0, 0, 0);
  in.total_sequence_length = 64;
  out.output = t4(NEXT(), GQA_F16, 3, 2, 1, 8 * 128, 0);
  out.present_key = t4(NEXT(), GQA_F16, 4, 2, 2, 64, 128);
  out.present_value = t4(NEXT(), GQA_F16, 4, 2, 2, 64, 128);
  in.past_key = out.present_key;
  in.past_value = out.present_value;
  size_t bytes = 0;
  if (gqa_workspace_size(h, &in, &out, &bytes) != GQA_OK || bytes == 0) {
    fprintf(stderr, "valid call rejected: %s\n", gqa_last_error());
    return 4;
  }
  gqa_plan_info info;
  if (gqa_describe_plan(h, &in, &out, &info) != GQA_OK || info.regime != GQA_REGIME_DECODE) return 5;

  /* A key of the wrong hidden size is an invalid argument, with a reason. */
  in.key = t4(NEXT(), GQA_F16, 3, 2, 1, 3 * 128, 0);
  if (gqa_workspace_size(h, &in, &out, &bytes) != GQA_ERR_INVALID_ARGUMENT) return 6;
  if (gqa_last_error() == NULL || gqa_last_error()[0] == '\0') return 7;
  gqa_destroy(h);
  printf("c abi host check: ok (workspace %zu bytes)\n", bytes);
  return 0;
}
