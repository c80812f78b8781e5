"""GB300-native routed MoE branch: top-k dispatch into an expert-major receive
buffer, per-token FP8 quantisation, a grouped gated-SiLU FP8 expert MLP on
tcgen05 tensor cores, and a weighted combine -- hand-written CUDA for sm_103a
behind a small C ABI (``include/moe.h``).  This package is the thin Python
binding over that library; PyTorch supplies device memory and streams only.
"""
from .api import *  # noqa: F401,F403
