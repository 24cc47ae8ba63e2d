"""GB300-native fused attention forward."""
