"""GB300-native MiniMax Sparse Attention (MSA) training kernels.

The compute path is the CUDA library ``libmsa.so`` (C-ABI declared in ``include/msa.h``); the
Python side only marshals arguments.  Importing the package does not load the library: the
binding loads it on first use and raises if it is missing.
"""
from .inputs import BLOCK, WORKLOADS, Workload, make_inputs, workload_seed  # noqa: F401

__all__ = ["BLOCK", "WORKLOADS", "Workload", "make_inputs", "workload_seed"]
