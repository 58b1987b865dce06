"""GB300-native slot-indexed recurrent-state cache for KDA/GDN linear-attention layers."""
