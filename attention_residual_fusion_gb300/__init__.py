"""GB300-native Kimi-K3 attention-residual (AttnRes) mixture."""
