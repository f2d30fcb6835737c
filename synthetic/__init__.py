"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke run.

This package only *draws* inputs (weights with a prescribed spectrum, latents,
queries) and rounds them to storage dtypes. It contains no decode-attention
arithmetic: neither the CUDA path nor the oracle lives here.
"""
from .gen import CONFIGS, Config, config_by_id, make_inputs, storage_round, hadamard_sylvester  # noqa: F401
