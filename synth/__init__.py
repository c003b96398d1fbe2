"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This package holds *only* input generation: counter-based random numbers
(splitmix64, Steele, Lea & Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), an Irwin-Hall approximation of N(0, 1) rounded to
bf16, the planted structure of the workloads (hot blocks, attention sink),
request lengths and the five workload recipes.  It contains none of the
token-dropping method's arithmetic (no attention, softmax, reduction,
selection or compaction), so importing it from either side couples nothing.

`synth.cpu` is a numpy implementation; `synth.gpu` drives a CUDA kernel that
produces bit-identical values directly in device memory, so that multi-GB
workloads never cross the host link.  Every value is a pure function of
(seed, tensor id, element index), so either side can regenerate any slice.
"""
from .recipe import CONFIGS, Workload, workload  # noqa: F401
