"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This package only *draws* inputs (weights with a prescribed spectrum, latents,
queries) and rounds them to storage dtypes. It contains no decode-attention
arithmetic: neither the CUDA path nor the oracle lives here.
"""
from .gen import (ABSORBED_FP16, ALL, ROPE_BF16, ROPE_FP16, ROPE_INT4, TINY_FP32, Config,  # noqa: F401
                  hadamard_sylvester, make_inputs, storage_round)
