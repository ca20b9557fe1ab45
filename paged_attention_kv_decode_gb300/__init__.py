"""GB300-native paged attention over a paged KV cache (binding loaded lazily)."""
