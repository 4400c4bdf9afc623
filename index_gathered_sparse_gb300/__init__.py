"""QSA gather-GQA sparse attention over a ragged, paged KV cache, for GB300.

The compute path is the C-ABI library ``libqsa.so`` (hand-written sm_103a CUDA
kernels); :mod:`.binding` marshals PyTorch tensors into it.  Nothing here
falls back to the CPU: a missing library raises.
"""
