"""GB300-native DSpark draft-sample / schedule / verify hot path.

The compute lives in libdspark.so (CUDA for sm_103a, C ABI in include/dspark.h);
this package holds the build step, the ctypes binding and the seeded workload
generators.
"""
from .binding import (DSparkError, draft_sample, load, read_device_flags, schedule_prefix, verify,
                      version, workspace_bytes)

__all__ = ["DSparkError", "draft_sample", "load", "read_device_flags", "schedule_prefix", "verify",
           "version", "workspace_bytes"]
