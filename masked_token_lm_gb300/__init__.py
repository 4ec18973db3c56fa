"""GB300-native mask-only logits (gather-GEMM) for diffusion-LLM inference.

The compute path is the C-ABI library ``libmosaic.so`` built from ``csrc/`` for sm_103a; the
Python layer (``mosaic``) only marshals arguments to it.
"""
__all__ = ["mosaic", "workloads"]
