"""GB300-native (sm_103a) Mamba2 SSD selective scan over packed varlen sequences.

The compute lives in ``libssd_scan.so`` (hand-written CUDA, C ABI in
``include/ssd_scan.h``); :mod:`.binding` marshals torch tensors into it.
"""
from .binding import (SSDError, ScanParams, call, kernel_path, load, make_params,  # noqa: F401
                      num_launches, ssd_scan_varlen, workspace_size)
from ._build import build  # noqa: F401
