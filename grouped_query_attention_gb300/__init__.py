"""GB300-native GroupQueryAttention forward pass (placeholder; binding added with the library)."""
