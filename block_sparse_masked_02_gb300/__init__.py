"""GB300-native (sm_103a) flash attention with a dynamic 4D mask (dense or
FlashMask column ranges), a learnable 4D bias, block skipping, and fused dBias."""
