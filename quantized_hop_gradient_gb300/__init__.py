"""GB300-native DynamiQ compressed multi-hop all-reduce (single-GPU simulation)."""
