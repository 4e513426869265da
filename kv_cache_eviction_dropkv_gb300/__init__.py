"""GB300-native (sm_103a) DropKV eviction-scoring path.

score -> select -> compact over device buffers, behind the C-ABI library
libdropkv.so (built from csrc/ by __graft_entry__.build()).  The Python layer
only marshals arguments; every step runs in the library's CUDA kernels.
"""
