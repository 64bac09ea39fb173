"""Seeded synthetic workloads shared by the oracle tests and the CUDA path (no method arithmetic)."""
from .workloads import *  # noqa: F401,F403
from .workloads import (WorkloadSpec, Workload, WORKLOADS, make_workload, f32_to_bf16_bits,
                        bf16_bits_to_f32, inject_mask_noise, spec_for)
