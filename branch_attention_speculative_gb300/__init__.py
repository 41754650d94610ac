"""Draft branch attention on one GB300 (sm_103a): causal main attention over
packed zigzag chunks + rank-local branch attention, merged by Eq. 2.

The compute path is libba.so (CUDA kernels behind a C ABI, ``include/ba.h``);
``api`` is a thin ctypes binding over it.  ``workloads`` draws seeded
synthetic inputs."""

from . import workloads  # noqa: F401

__all__ = ["workloads", "api", "build"]
