"""GB300-native (sm_103a) gated delta rule: chunkwise forward, decode step
and the output epilogue (RMSNorm + SiLU output gate).

The computation lives in ``libgdr.so`` (hand-written CUDA kernels behind the C
ABI of ``include/gdr.h``); this package only marshals arguments to it.
"""
from ._binding import (BETA_CHANNEL, CHUNK, DECAY_CHANNEL, ERASE_CHANNEL, GDR_BF16, GDR_F32, QMIX,
                       WRITE_CHANNEL, GdrError, Shape, chunk_bwd, chunk_bwd_check, chunk_bwd_workspace_bytes, token_bwd, token_bwd_workspace_bytes, chunk_fwd, chunk_fwd_check, chunk_fwd_workspace_bytes,
                       chunk_fwd_pipelined_workspace_bytes, gate_cumsum, lib, make_shape,
                       pipeline_segments, recurrent_step, rmsnorm_gate, status_string,
                       token_fwd)

__all__ = ["BETA_CHANNEL", "CHUNK", "DECAY_CHANNEL", "ERASE_CHANNEL", "WRITE_CHANNEL", "QMIX", "GDR_BF16",
           "GDR_F32", "GdrError", "Shape", "chunk_bwd", "chunk_bwd_check", "chunk_bwd_workspace_bytes", "token_bwd", "token_bwd_workspace_bytes", "chunk_fwd", "chunk_fwd_check", "chunk_fwd_workspace_bytes",
           "chunk_fwd_pipelined_workspace_bytes", "gate_cumsum", "lib", "make_shape",
           "pipeline_segments", "recurrent_step", "rmsnorm_gate", "status_string", "token_fwd"]
