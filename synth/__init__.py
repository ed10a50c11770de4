"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This package draws random numbers and rounds them to the storage dtype; it
performs none of the attention arithmetic.  See ``synth.inputs``.
"""
from .inputs import (CONFIGS, Workload, make_omega_orf, make_omega_iid,
                     make_qkv, make_workload, make_upstream_grad, round_bf16)

__all__ = ["CONFIGS", "Workload", "make_omega_orf", "make_omega_iid",
           "make_qkv", "make_workload", "make_upstream_grad", "round_bf16"]
