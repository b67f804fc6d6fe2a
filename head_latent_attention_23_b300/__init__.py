"""B300-native Multi-Head Latent Attention decode.

The compute path is the C-ABI library ``libmla.so`` (hand-written CUDA for
sm_103a); ``head_latent_attention_23_b300.mla`` is its thin Python binding.
Importing this package loads nothing; the library is loaded on first use and
the call fails loudly if it is missing.
"""
__all__ = ["mla", "workloads"]
