"""GB300-native MoE token dispatch / combine.

The computation lives in hand-written sm_103a CUDA kernels behind the C ABI of
include/moe.h (libcrs_moe.so); ``combine_route_scan_gb300.moe`` is the thin
Python binding over it. PyTorch supplies device memory and streams only.
"""
