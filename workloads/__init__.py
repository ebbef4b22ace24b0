"""Seeded synthetic workloads shared (as data only) by the oracle tests, the
CUDA parity tests and the benchmark."""
from .gen import (Workload, make, CONFIGS, tiny, distinct_decode, zipf_decode,
                  sparse_prefill, rank_sweep, make_custom, algorithmic_bytes,
                  f32_to_bf16_bits, bf16_bits_to_f32)
