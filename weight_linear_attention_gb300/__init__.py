"""GB300 (sm_103a) Falcon fast-weight attention: chunk-parallel forward scan.

The compute path is the C-ABI library ``_build/libfalcon.so`` (CUDA kernels);
``falcon`` is its ctypes binding, ``inputs`` the seeded synthetic workloads,
``build`` the nvcc build. Importing this package loads nothing; the library is
opened on first use.
"""

__all__ = ["falcon", "inputs", "build"]
