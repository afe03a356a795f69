"""GB300 (sm_103a) hot path of LoCo low-bit gradient compression.

``bit_gradient_compression_gb300.loco``  binding of libloco (include/loco.h)
``bit_gradient_compression_gb300.build`` in-tree nvcc build of libloco.so
``bit_gradient_compression_gb300.workloads`` seeded synthetic gradient buckets

The binding is imported on first use so that the workload generators and the
build script work on a machine where the library has not been built yet.
"""

__all__ = ["loco", "build", "workloads"]
