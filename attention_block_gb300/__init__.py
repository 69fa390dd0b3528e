"""GB300-native fused decode attention block (placeholder; binding follows)."""
