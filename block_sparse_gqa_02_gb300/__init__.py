"""MiniMax Sparse Attention (MSA) hot path for GB300 (sm_103a)."""
