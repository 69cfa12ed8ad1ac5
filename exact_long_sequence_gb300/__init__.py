"""GB300-native exact self-attention forward (placeholder; binding follows)."""
