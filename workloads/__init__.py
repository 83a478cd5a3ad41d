"""Seeded synthetic inputs for the speculative-decoding draft/verify path.

This package only draws random numbers and lays them out; it holds none of
the method's arithmetic (no softmax, top-k, tree, acceptance or sampling).
Both the CUDA path and the CPU oracle take their inputs from here.
"""
from .synth import CONFIGS, Cfg, assemble_target, generate, step_offsets

__all__ = ["CONFIGS", "Cfg", "assemble_target", "generate", "step_offsets"]
