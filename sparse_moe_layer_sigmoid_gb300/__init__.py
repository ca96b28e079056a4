"""LatentMoE layer forward pass on GB300 (sm_103a): Python binding over the C-ABI library."""
