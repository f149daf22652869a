"""GB300-native (sm_103a) Mamba2 SSD selective scan over packed varlen sequences.

The compute lives in ``libssd_scan.so`` (hand-written CUDA, C ABI in
``include/ssd_scan.h``); :mod:`.binding` marshals torch tensors into it.
"""
from .binding import (ReplayParams, SSDError, ScanParams, call, call_noalloc,  # noqa: F401
                      call_replay, kernel_path, load, make_params, make_replay_params,
                      num_launches, ssd_scan_varlen, workspace_size)
from ._build import build  # noqa: F401
