"""GB300-native (sm_103a) Mamba2 SSD selective scan over packed varlen sequences.

The compute lives in ``libssd_scan.so`` (hand-written CUDA, C ABI in
``include/ssd_scan.h``); :mod:`.binding` marshals torch tensors into it.
"""
from .binding import (SSDError, ScanParams, call, call_noalloc, kernel_path, load,  # noqa: F401
                      make_params,
                      num_launches, ssd_scan_varlen, workspace_size)
from ._build import build  # noqa: F401
