"""CPU oracle for the MoE-layer expert-cache path.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()`` and
by the CPU-baseline leg of ``bench.py``; never by the library.
"""
from .moe import *  # noqa: F401,F403
from .moe import (FT_CPU, Counters, SlotCache, StepRecord, all_pair_rows, bf16_to_f64, combine,
                  decode_layer_outputs, dedupe, e4m3_to_f64, matvec_post_scaled, mbps, pair_row,
                  prefill_outputs, rel_err_rows, route, router_logits, silu, split_misses, swiglu_expert,
                  GATE_SOFTMAX_TOPK, GATE_SOFTMAX_ALL, GATE_SIGMOID_TOPK, E2M1_TABLE, e2m1_unpack_to_f64,
                  matvec_nvfp4, NVFP4_BLOCK, e8m0_to_f64, matvec_mxfp4, MXFP4_BLOCK)
