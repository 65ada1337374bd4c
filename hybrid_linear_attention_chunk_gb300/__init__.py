"""KDA (Kimi Delta Attention) chunked prefill and decode step on one GB300.

The compute path is libkda.so, a C-ABI library of hand-written sm_103a CUDA
kernels (declared in include/kda.h).  This package holds its build script,
its ctypes binding (same names as the C entry points) and the seeded
synthetic input generator.  Importing the package does not load the library;
the first call does, and raises if it is missing.
"""
from ._lib import (KdaChunkDesc, KdaDecodeDesc, KdaError, KdaLayerGates, chunk_desc, kda_chunk_fwd,  # noqa: F401
                   kda_affine_compose, kda_chunk_affine_pair,
                   kda_chunk_bwd, kda_chunk_bwd_workspace_size, kda_chunk_fwd_ckpt, kda_chunk_fwd_noalloc,
                   kda_chunk_fwd_workspace_size, kda_decode_step,
                   kda_layer_decode_step, kda_layer_fwd, layer_gates, load, LIB_PATH)
from .cp import kda_chunk_fwd_cp  # noqa: F401

__all__ = ["kda_chunk_fwd", "kda_chunk_affine_pair", "kda_affine_compose", "kda_chunk_fwd_cp", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size", "kda_chunk_fwd_ckpt", "kda_chunk_fwd_noalloc", "kda_decode_step",
           "kda_layer_fwd", "kda_layer_decode_step", "kda_chunk_fwd_workspace_size", "load", "KdaError",
           "KdaChunkDesc", "KdaDecodeDesc", "KdaLayerGates", "chunk_desc", "layer_gates", "LIB_PATH"]
