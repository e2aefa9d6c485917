"""Seeded synthetic input generators (shared by the oracle and the GPU tests)."""
from .inputs import (Problem, TILE, HEAD_DIM, bf16_bits_from_f32, bf16_bits_to_f32,  # noqa: F401
                     config, packed, sequence, small, varlen_lengths)
