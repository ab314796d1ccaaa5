"""GB300-native small-M routed-MoE decode/verify layer (see include/moe.h)."""
