"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

Holds no loss arithmetic: only random draws shaped into logits, targets, masks,
planted margins and packed segments.
"""
from .workloads import (  # noqa: F401
    IGNORE_INDEX, ORDER, WORKLOADS, Workload, bf16_round, build, get, normal_1d,
    permutation, philox_kat, randint_1d, uniform_1d,
)
