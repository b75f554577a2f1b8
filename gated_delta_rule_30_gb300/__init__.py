"""GB300-native Kimi Delta Attention forward pass (binding filled in below)."""
