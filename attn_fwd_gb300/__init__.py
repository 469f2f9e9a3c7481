"""GB300-native exact attention: tiled forward with online softmax and a
recompute backward, as hand-written sm_103a CUDA behind a C ABI (libfa.so).

The binding in :mod:`attn_fwd_gb300.fa` marshals PyTorch tensors into the C
calls; every arithmetic step runs in the library's kernels.
"""
