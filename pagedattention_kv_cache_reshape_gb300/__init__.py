"""GB300-native paged KV-cache write and paged attention (C-ABI library + binding)."""
