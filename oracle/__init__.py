"""CPU oracle for the MoE routed branch (dispatch -> FP8 quant -> gated-SiLU
expert MLP -> weighted combine).

TEST INFRASTRUCTURE ONLY.  Nothing in the product package may import this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.  It shares no code, table or helper with the CUDA path.

Sources (page title, then the section on that page):

* "SGLang、NCCL 与 MoE EP" -- Level 1 §1.1 (the MoE output and where the router
  weight is applied), §2.1 (expert placement), §2.3.1-2.3.7 (source tensors,
  receive and compact, counters and the source map), §3.2 and §3.4 (the traced
  token and the replay), §5.3 (byte and FLOP accounting).
* "SGLang Expert Compute Backend" -- §1.1 (gated MLP), §2.4 (tiles), §3.5
  (block-wise FP8 scale math and addressing), §3.6-3.7 (activation, requant,
  down projection, output view), §4.3 (BM table), §5.3-5.4 (split and fill rate).
* "DeepEP 架构与实现笔记" -- §11 (the per-token FP8 cast rule) and §9.6 (combine
  applies the router weights in a weighted reduce).
"""
from .moe_oracle import *  # noqa: F401,F403
