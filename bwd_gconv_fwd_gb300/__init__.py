"""GB300-native grouped 2D convolution (NCHW)."""
