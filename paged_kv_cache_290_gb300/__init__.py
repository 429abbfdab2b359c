"""GB300 (sm_103a) paged attention: KV scatter-write and block-table-indirected attention.

The compute runs in the CUDA library ``libpa_gb300.so`` (C ABI in ``include/pa.h``); the
names exported here are its thin Python binding.  ``workloads`` holds the seeded synthetic
inputs used by tests and the benchmark.
"""
from .binding import (PAError, BatchDescriptor, attention, get_device_error, last_error,
                      load_library, reshape_and_cache, set_timing_events, version,
                      workspace_size)

__all__ = ["PAError", "BatchDescriptor", "attention", "get_device_error", "last_error",
           "load_library", "reshape_and_cache", "set_timing_events", "version",
           "workspace_size"]
