// Launch interface between the C ABI (gdr_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace gdr {

constexpr int kChunkLen = 64;  // C, the chunk length of the WY/UT algorithm

// Arguments of the chunkwise forward; pointers as documented in include/gdr.h.
struct ChunkArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* lam;
  const void* b;
  const void* w;
  const float* h0;
  void* o;
  float* hT;
  int B, T, H, dv;
  unsigned flags;
  float scale;
  // output epilogue fused into the state pass (transposed scan only): with gz
  // non-null, o receives y = o rsqrt(mean(o^2) + geps) gw silu(gz) per
  // (token, head) row instead of o
  const void* gz = nullptr;
  const float* gw = nullptr;
  float geps = 0.f;
};

// Arguments of the single-token recurrent step.
struct StepArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;
  const float* beta;
  const float* lam;
  const void* b;
  const void* w;
  float* state;
  void* o;
  int N, H;
  unsigned flags;
  float scale;
};

// Arguments of the token-order scan with a write strength per value channel.
struct ValueBetaArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* g;      // [B, T, H] log-decay
  const float* beta;   // [B, T, H, d_v]
  const float* h0;     // [B, H, d_k, d_v] or null (zero state)
  void* o;
  float* hT;           // [B, H, d_k, d_v] or null; may equal h0
  int B, T, H;
  float scale;
};

// Device status words the tensor-core chunk kernel reports into (in the
// caller's workspace): [0] = 0 or a gdr_status code, [1] = CTA index,
// [2] = 4 * chunk + which wait gave up.
constexpr int kStatusWords = 4;
constexpr size_t kChunkWorkspaceBytes = 256;

// fp32 inputs: split-precision warp-MMA kernel (value slice width chosen
// inside). bf16 inputs: tcgen05 kernel, 64-wide value slices.
cudaError_t launch_chunk_fwd_f32(const ChunkArgs& a, int dk, cudaStream_t stream);
cudaError_t launch_chunk_fwd_tc(const ChunkArgs& a, int dk, int* status, cudaStream_t stream);

// bf16 inputs with scalar gates (no channel decay, erase or write gate): the
// pipelined TMA + tcgen05 kernel; tq, tk, tv from make_bthd_tmap.
bool chunk_fwd_pipe_supports(unsigned flags);
cudaError_t launch_chunk_fwd_pipe(const ChunkArgs& a, int dk, const CUtensorMap& tq,
                                  const CUtensorMap& tk, const CUtensorMap& tv, int* status,
                                  cudaStream_t stream);
// bf16 inputs, two-kernel path: the chunk preparation kernel writes one packet
// per chunk (packet.h) into `packets`, then the chunk scan kernel runs the
// state pass over them. `packets` holds B * H * ceil(T / 64) packets.
// PrepRange limits the preparation to chunks chunk0 .. chunk0 + chunks - 1 of
// every (batch, head) (chunks 0: to the end). With a counter (an int that
// reads 0 when the launch starts), CTAs claim the chunks one at a time, at
// most per_cta each, instead of a fixed persistent stride.
struct PrepRange {
  int chunk0 = 0;
  int chunks = 0;
  int* counter = nullptr;
  int per_cta = 0;
};
cudaError_t launch_chunk_prep(const ChunkArgs& a, int dk, unsigned char* packets, int* status,
                              cudaStream_t stream, const PrepRange& rg = PrepRange());
// the claimed-work variant (rg.counter non-null), which launch_chunk_prep calls
cudaError_t launch_chunk_prep_claimed(const ChunkArgs& a, int dk, unsigned char* packets,
                                      int* status, cudaStream_t stream, const PrepRange& rg);
// Sequence split of the scan: `segments` runs of `seg_chunks` chunks per
// (batch, head) from chunk `chunk0` on (seg_chunks 0: one run of every chunk
// from chunk0). States per run are
// [B, H, segments, d_k, width] fp32. h0_per_seg: a.h0 holds one start state
// per run (else a.h0, [B, H, d_k, d_v], starts run 0 and the others start at
// zero). hT_per_seg: every run writes its end state to a.hT (else only the
// last run writes a.hT, [B, H, d_k, d_v]). hT_hom non-null adds d_k / 64
// identity slices per run whose end states (each run's transition, d_k x d_k)
// go there.
struct ScanSegments {
  int segments = 1;
  int seg_chunks = 0;
  int chunk0 = 0;          // the first run starts at this chunk
  bool h0_per_seg = false;
  bool hT_per_seg = false;
  float* hT_hom = nullptr;
};
cudaError_t launch_chunk_scan(const ChunkArgs& a, int dk, const unsigned char* packets,
                              int* status, cudaStream_t stream,
                              const ScanSegments& sg = ScanSegments());
// d_k = d_v = 128 without the per-value-channel write strength: the state pass
// runs transposed (chunk_scan_t.cu), one CTA per (batch, head), and the packets
// hold U^T instead of U.
inline bool scan_transposed(int dk, int dv, unsigned flags) {
  return dk == 128 && dv == 128 && !(flags & 16u);
}
cudaError_t launch_chunk_scan_t(const ChunkArgs& a, int dk, const unsigned char* packets,
                                int* status, cudaStream_t stream, ScanSegments sg);
// S_start[p] = M[p-1] S_start[p-1] + H[p-1] over the runs of each (batch,
// head), S_start[0] = h0 (or zero): M [B,H,P,d_k,d_k], Hl and S [B,H,P,d_k,d_v].
cudaError_t launch_segment_combine(const float* M, const float* Hl, const float* h0, float* S,
                                   int B, int H, int P, int dk, int dv, cudaStream_t stream);
cudaError_t launch_recurrent_step(const StepArgs& a, int dk, int dv, bool f32,
                                  cudaStream_t stream);
// Output epilogue over `rows` rows of d_v channels (dv 64, 128 or 256):
// y = o rsqrt(mean(o^2) + eps) weight silu(z); fp32 or bf16 rows, fp32 weight.
cudaError_t launch_rmsnorm_gate(const void* o, const void* z, const float* weight, float eps,
                                void* y, long long rows, int dv, bool f32,
                                cudaStream_t stream);
// Chunkwise backward (every flag but 16): fp32 records in the workspace,
// chunk_bwd_workspace_bytes of it; gradients are fp32 in the inputs' layouts.
struct ChunkBwdArgs {
  const void *q, *k, *v, *dO;
  const float *g, *beta, *lam;
  const void *b, *w;
  const float *h0, *dhT;
  float *dq, *dk, *dv, *dg, *dbeta, *dlam, *db, *dw, *dh0;
  void* workspace;
  int B, T, H, dk_dim, dv_dim;
  unsigned flags;
  float scale;
};
size_t chunk_bwd_workspace_bytes(int B, int T, int H, int dk, int dv);
cudaError_t launch_chunk_bwd(const ChunkBwdArgs& a, bool f32, cudaStream_t stream);
// The same gradients walked token by token (every flag but 16; no decay
// factoring, so no range limit): token_bwd_workspace_bytes of workspace,
// d_v a multiple of 16; dq, dk, dg, db, dbeta and dlam are summed with atomics
// into outputs the launch zeroes first.
size_t token_bwd_workspace_bytes(int B, int T, int H, int dk, int dv);
cudaError_t launch_token_bwd(const ChunkBwdArgs& a, bool f32, cudaStream_t stream);

// Token-order scan for every flag but 16 (no decay factoring: the path past the
// chunked path's channel-decay range); o and hT as in the chunked forward.
cudaError_t launch_token_scan(const ChunkArgs& a, int dk, bool f32, cudaStream_t stream);
// Write strength per value channel (flag 16): token-order scan, fp32 state.
cudaError_t launch_value_beta_scan(const ValueBetaArgs& a, int dk, int dv, bool f32,
                                   cudaStream_t stream);
// Gradients of the token-order scan with a write strength per value channel
// (flag 16): inputs as ValueBetaArgs plus dO (the call's dtype) and dhT (fp32,
// or null); fp32 outputs dq, dk [B,T,H,nk], dv, dbeta [B,T,H,nv], dg [B,T,H],
// dh0 [B,H,nk,nv] (or null); value_beta_bwd_workspace_bytes of workspace
// (16-byte aligned). nv must be a multiple of 32.
struct ValueBetaBwdArgs {
  const void *q, *k, *v, *dO;
  const float *g, *beta, *h0, *dhT;
  float *dq, *dk, *dv, *dg, *dbeta, *dh0;
  void* workspace;
  int B, T, H, nk, nv;
  float scale;
};
size_t value_beta_bwd_workspace_bytes(int B, int T, int H, int dk, int dv);
cudaError_t launch_value_beta_bwd(const ValueBetaBwdArgs& a, bool f32, cudaStream_t stream);
cudaError_t launch_gate_cumsum(const float* g, float* G, int B, int T, int X,
                               cudaStream_t stream);

}  // namespace gdr
