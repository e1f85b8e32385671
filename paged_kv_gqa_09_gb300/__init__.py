"""paged_kv_gqa_09_gb300 -- paged-KV grouped-query decode attention for GB300.

A GB300-native (sm_103a) implementation of the decode engine of "PersistentKV:
Page-Aware Decode Scheduling for Long-Context LLM Serving on Commodity GPUs":
attention read straight through the block table, sequence splitting with an
exact log-sum-exp merge, row-local bounds, a compact device-built workqueue and
a calibrated path policy.  The kernels and the C ABI live in libpkv.so
(include/pkv.h); this package is its Python binding.
"""
from .build import build as build_library  # noqa: F401
from ._lib import (PKV_OK, PKV_EINVAL, PKV_EUNSUPPORTED, PKV_ECUDA, PKV_EDEVICE,  # noqa: F401
                   PKV_ETIMEOUT, PKV_ECAPACITY, PKV_PATH_BUCKETED_SPLIT, PKV_PATH_WORKQUEUE,
                   PKV_PATH_SINGLE_PASS, PATH_EXACT_BUCKETS, PkvError, PkvLibraryError)
from .api import *  # noqa: F401,F403
