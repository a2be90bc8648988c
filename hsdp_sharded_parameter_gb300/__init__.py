"""GB300-native HSDP fully_shard parameter and gradient data path.

All rank_size virtual ranks live in one GPU's HBM; the shard-group
ReduceScatter, the replicate-group AllReduce and the AllGather become
on-device kernels (hand-written CUDA for sm_103a) behind a C-ABI library.
The Python layer (``capi``) only marshals arguments into that library.
"""
__all__ = ["capi", "workloads"]
