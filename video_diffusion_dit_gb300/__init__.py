"""GB300 (sm_103a) SANA-Video linear attention over rotated queries and keys.

``video_diffusion_dit_gb300.lin_attn`` is the Python binding of the C-ABI
library (``liblin_attn.so``); importing it fails loudly if the library has not
been built.  ``video_diffusion_dit_gb300.synth`` makes seeded synthetic inputs.
"""
__all__ = ["lin_attn", "synth"]
