"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

Holds no addressing or attention arithmetic (see ``workloads``)."""
from .workloads import (BF16_NAN_BITS, WORKLOADS, Draw, Workload, bf16_bits, draw, draw_explicit,
                        draw_mla_write, values)

__all__ = ["BF16_NAN_BITS", "WORKLOADS", "Draw", "Workload", "bf16_bits", "draw", "draw_explicit",
           "draw_mla_write", "values"]
