"""fp8 (E4M3) paged KV cache for GB300: quantise-on-append and paged decode
attention, as the C-ABI library libfp8kv with a thin Python binding.

Importing this package does not load the native library; the first call of a
binding function does, and it raises if the library is missing.
"""
