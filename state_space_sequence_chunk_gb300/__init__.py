"""GB300-native Mamba-2 SSD chunked-scan forward pass."""
