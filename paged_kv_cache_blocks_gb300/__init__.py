"""GB300-native paged KV-cache decode (PagedAttention) behind a C ABI."""
