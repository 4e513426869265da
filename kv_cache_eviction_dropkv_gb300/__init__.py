"""GB300-native (sm_103a) DropKV eviction-scoring path.

score -> select -> compact over device buffers, behind the C-ABI library
libdropkv.so (built from csrc/ by __graft_entry__.build()).  The Python layer
only marshals arguments; every step runs in the library's CUDA kernels.
"""
from ._binding import (DropKVError, dropkv_compact, dropkv_read_status, dropkv_score, dropkv_select,  # noqa: F401
                       dropkv_shape, dropkv_version, dropkv_workspace_size, make_shape)
from .api import DropKV  # noqa: F401
