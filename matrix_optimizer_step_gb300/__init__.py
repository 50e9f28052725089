"""GB300-native owner-side Muon / AdamW optimizer step.

The product is ``libdmuon.so`` (CUDA kernels for sm_103a behind the C ABI
of ``include/dmuon.h``); this package is its thin Python binding:

* ``capi``       ctypes wrappers named after the C entry points;
* ``optim``      ``OwnerStep``, a context plus cached descriptor arrays;
* ``workloads``  seeded synthetic inputs and work accounting;
* ``build``      the nvcc build of the library.

Importing the package does not load the library; the first call does, and
raises if it has not been built.
"""

from .capi import (  # noqa: F401
    DMUON_DTYPE_BF16,
    DMUON_DTYPE_F32,
    DMUON_FLAG_FP32_NS,
    DMUON_FLAG_NESTEROV,
    DmuonError,
    dmuon_adamw_step,
    dmuon_context_create,
    dmuon_context_destroy,
    dmuon_context_set_tuning,
    dmuon_kernel_launches,
    dmuon_lpt_assign,
    dmuon_lpt_assign_layered,
    dmuon_muon_step,
    dmuon_muon_step_noalloc,
    dmuon_muon_step_noalloc_sync,
    dmuon_profile,
    dmuon_profile_read,
    dmuon_selftest_wait_timeout,
    dmuon_set_tuning,
    dmuon_status_string,
    dmuon_step_host,
    dmuon_sync,
    load_library,
)
from .optim import OwnerStep, adamw_shard_ranges, adamw_shard_views, owner_partition  # noqa: F401
