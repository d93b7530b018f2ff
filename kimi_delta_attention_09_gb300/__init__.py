"""GB300-native Kimi Delta Attention (KDA) hot path: chunked prefill and paged decode."""
