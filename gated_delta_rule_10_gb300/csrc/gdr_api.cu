// The C ABI of the library (declared in include/gdr.h): argument checks and
// kernel dispatch. Nothing here allocates memory; only gdr_chunk_fwd_check
// synchronises the stream.
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <limits>

#include "gdr.h"
#include "kernels.h"
#include "packet.h"
#include "tma.h"

namespace {

constexpr int kAbiVersion = 2;
constexpr long long kMaxElems = std::numeric_limits<int>::max();

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

gdr_status check_shape(const gdr_shape* s, bool step) {
  if (!s) return GDR_ERR_INVALID_ARG;
  if (s->B < 1 || s->T < 1 || s->H < 1 || s->dk < 1 || s->dv < 1) return GDR_ERR_INVALID_ARG;
  if (s->dtype != GDR_F32 && s->dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
  if (s->flags & ~31u) return GDR_ERR_INVALID_ARG;
  // the write strength per value channel comes with one scalar decay per head
  // and no other gate
  if ((s->flags & GDR_BETA_CHANNEL) && (s->flags & 15u)) return GDR_ERR_UNSUPPORTED;
  if (!std::isfinite(s->scale)) return GDR_ERR_INVALID_ARG;
  if (step && s->T != 1) return GDR_ERR_INVALID_ARG;
  if ((s->dk != 64 && s->dk != 128) || (s->dv != 64 && s->dv != 128)) return GDR_ERR_UNSUPPORTED;
  const long long d = s->dk > s->dv ? s->dk : s->dv;
  const long long elems = static_cast<long long>(s->B) * s->T * s->H * d;
  const long long state = static_cast<long long>(s->B) * s->H * s->dk * s->dv;
  if (elems > kMaxElems || state > kMaxElems) return GDR_ERR_UNSUPPORTED;
  if (s->H > 65535 || s->B > 65535) return GDR_ERR_UNSUPPORTED;  // grid y / z extents
  if ((s->flags & GDR_BETA_CHANNEL) && static_cast<long long>(s->B) * s->H > 65535)
    return GDR_ERR_UNSUPPORTED;                                     // grid y extent
  return GDR_OK;
}

// Pointer rules shared by the chunked forward and the recurrent step.
gdr_status check_gates(const gdr_shape* s, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* lam, const void* b,
                       const void* w, const void* o) {
  const unsigned f = s->flags;
  if (!q || !k || !v || !g || !o) return GDR_ERR_INVALID_ARG;
  const bool need_beta = !((f & GDR_ERASE_CHANNEL) && (f & GDR_WRITE_CHANNEL));
  if (need_beta && !beta) return GDR_ERR_INVALID_ARG;
  if ((f & GDR_QMIX) && !lam) return GDR_ERR_INVALID_ARG;
  if ((f & GDR_ERASE_CHANNEL) && !b) return GDR_ERR_INVALID_ARG;
  if ((f & GDR_WRITE_CHANNEL) && !w) return GDR_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return GDR_ERR_INVALID_ARG;
  if (!aligned(g, 4) || (beta && !aligned(beta, 4)) || (lam && !aligned(lam, 4)))
    return GDR_ERR_INVALID_ARG;
  if ((f & GDR_DECAY_CHANNEL) && !aligned(g, 16)) return GDR_ERR_INVALID_ARG;   // vector loads
  if ((f & GDR_ERASE_CHANNEL) && !aligned(b, 16)) return GDR_ERR_INVALID_ARG;
  if ((f & GDR_WRITE_CHANNEL) && !aligned(w, 16)) return GDR_ERR_INVALID_ARG;
  if ((f & GDR_BETA_CHANNEL) && !aligned(beta, 16)) return GDR_ERR_INVALID_ARG;
  return GDR_OK;
}

// Sequence split of the two-kernel path (bf16, every flag but BETA_CHANNEL).
constexpr int kSplitTargetCtas = 152;   // one wave of scan CTAs on a GB300
constexpr int kSplitMinChunks = 8;      // chunks per run, at least

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int n_chunks_of(const gdr_shape* s) { return (s->T + gdr::kChunkLen - 1) / gdr::kChunkLen; }

bool split_allowed(const gdr_shape* s) {
  return s->dtype == GDR_BF16 && !(s->flags & GDR_BETA_CHANNEL);
}

// Runs per (batch, head) that the default path uses. The scan walks the chunks
// of each (batch, head) in order, so when B * H leaves SMs idle the sequence is
// cut into P runs. Cost in chunk steps of one scan CTA (about 1.3 us at 2 GHz):
// unsplit, waves of the value CTAs times the chunks; split, the first pass
// (value and identity slices) and the last pass each over one run, plus about
// 4 steps per run for chaining the start states and 10 for the extra launches.
// P is the power of two with the least cost among those whose first pass fits
// one wave (a second wave measured slower per step than the model says) and
// whose runs hold at least kSplitMinChunks chunks.
int default_segments(const gdr_shape* s) {
  if (!split_allowed(s)) return 1;
  const long long bh = static_cast<long long>(s->B) * s->H;
  const long long val = bh * (s->dv / 64), both = bh * ((s->dv + s->dk) / 64);
  const long long nc = n_chunks_of(s);
  const double unsplit =
      static_cast<double>((val + kSplitTargetCtas - 1) / kSplitTargetCtas * nc);
  double best = unsplit;
  int best_p = 1;
  for (int P = 2; P * both <= kSplitTargetCtas && static_cast<long long>(P) * kSplitMinChunks <= nc;
       P *= 2) {
    const long long per = (nc + P - 1) / P;
    const double cost = 2.0 * per + 4.0 * P + 10.0;
    if (cost < best) {
      best = cost;
      best_p = P;
    }
  }
  return best_p;
}

// runs actually used for a request of P: every run non-empty
void split_geometry(const gdr_shape* s, int P, int* runs, int* seg_chunks) {
  const int nc = n_chunks_of(s);
  const int per = (nc + P - 1) / P;
  *seg_chunks = per;
  *runs = (nc + per - 1) / per;
}

size_t two_kernel_bytes(const gdr_shape* s) {
  const size_t chunks = static_cast<size_t>(s->B) * s->H * static_cast<size_t>(n_chunks_of(s));
  const size_t per = (s->flags & GDR_BETA_CHANNEL) ? gdr::packet_vb_bytes(s->dk, s->dv)
                                                   : gdr::packet_bytes(s->dk, s->dv);
  return gdr::kChunkWorkspaceBytes + chunks * per;
}

// status words, packets, then per-run local end states, transitions and start states
size_t split_bytes(const gdr_shape* s, int P) {
  if (P <= 1) return two_kernel_bytes(s);
  const size_t runs = static_cast<size_t>(s->B) * s->H * P;
  const size_t st = runs * s->dk * s->dv * sizeof(float), tr = runs * s->dk * s->dk * sizeof(float);
  return align256(two_kernel_bytes(s)) + align256(st) + align256(tr) + align256(st);
}

gdr::ValueBetaArgs value_beta_args(const gdr_shape* s, const void* q, const void* k,
                                   const void* v, const float* g, const float* beta,
                                   const float* h0, void* o, float* hT) {
  gdr::ValueBetaArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = h0; a.o = o; a.hT = hT;
  a.B = s->B; a.T = s->T; a.H = s->H; a.scale = s->scale;
  return a;
}

}  // namespace

extern "C" {

int gdr_abi_version(void) { return kAbiVersion; }

const char* gdr_status_string(gdr_status status) {
  switch (status) {
    case GDR_OK: return "GDR_OK";
    case GDR_ERR_INVALID_ARG: return "GDR_ERR_INVALID_ARG: null or misaligned pointer, bad size or flag";
    case GDR_ERR_UNSUPPORTED: return "GDR_ERR_UNSUPPORTED: request outside the supported set";
    case GDR_ERR_CUDA: return "GDR_ERR_CUDA: the CUDA runtime reported an error";
    case GDR_ERR_WORKSPACE: return "GDR_ERR_WORKSPACE: workspace missing or too small";
    case GDR_ERR_TIMEOUT: return "GDR_ERR_TIMEOUT: a bounded device-side wait gave up";
    case GDR_ERR_RANGE:
      return "GDR_ERR_RANGE: a chunk's summed channel log-decay is below the chunked path's limit";
  }
  return "unknown gdr_status";
}

gdr_status gdr_chunk_fwd_workspace(const gdr_shape* shape, size_t* bytes) {
  if (!bytes) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  // bf16: the status words, then one packet per chunk of every (batch, head)
  // for the two-kernel path, and the run states when the sequence is split;
  // fp32 needs nothing
  if (shape->dtype != GDR_BF16) {
    *bytes = 0;
    return GDR_OK;
  }
  *bytes = split_allowed(shape) ? split_bytes(shape, default_segments(shape))
                                : two_kernel_bytes(shape);
  return GDR_OK;
}

gdr_status gdr_chunk_fwd_workspace_min(const gdr_shape* shape, size_t* bytes) {
  if (!bytes) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  *bytes = (shape->dtype == GDR_BF16 && !(shape->flags & GDR_BETA_CHANNEL))
               ? gdr::kChunkWorkspaceBytes
               : 0;
  return GDR_OK;
}

gdr_status gdr_chunk_fwd_workspace_split(const gdr_shape* shape, int segments, size_t* bytes) {
  if (!bytes || segments < 1) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  if (!split_allowed(shape)) {
    if (segments > 1) return GDR_ERR_UNSUPPORTED;
    *bytes = shape->dtype == GDR_BF16 ? two_kernel_bytes(shape) : 0;
    return GDR_OK;
  }
  *bytes = split_bytes(shape, segments);
  return GDR_OK;
}

}  // extern "C"

namespace {

// Status words a chunked call left at the start of its workspace.
gdr_status read_status(const void* workspace, gdr_stream_t stream, int* detail) {
  if (!workspace || !aligned(workspace, 16)) return GDR_ERR_INVALID_ARG;
  int words[gdr::kStatusWords] = {0, 0, 0, 0};
  const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(words, workspace, sizeof(words), cudaMemcpyDeviceToHost, st_) !=
          cudaSuccess ||
      cudaStreamSynchronize(st_) != cudaSuccess)
    return GDR_ERR_CUDA;
  if (detail) {
    detail[0] = words[1];
    detail[1] = words[2];
  }
  return words[0] == 0 ? GDR_OK : static_cast<gdr_status>(words[0]);
}

// The output epilogue's arguments: valid, and y apart from z.
gdr_status check_out_gate(const gdr_shape* s, const gdr_out_gate* gate, const void* y) {
  if (!gate || !gate->z || !gate->weight) return GDR_ERR_INVALID_ARG;
  if (!aligned(gate->z, 16) || !aligned(gate->weight, 16)) return GDR_ERR_INVALID_ARG;
  if (!std::isfinite(gate->eps) || gate->eps < 0.f) return GDR_ERR_INVALID_ARG;
  if (s->dv != 64 && s->dv != 128) return GDR_ERR_UNSUPPORTED;
  const uintptr_t bytes = static_cast<uintptr_t>(s->B) * s->T * s->H * s->dv *
                          (s->dtype == GDR_F32 ? 4 : 2);
  const uintptr_t py = reinterpret_cast<uintptr_t>(y), pz = reinterpret_cast<uintptr_t>(gate->z);
  if (pz < py + bytes && py < pz + bytes) return GDR_ERR_INVALID_ARG;
  return GDR_OK;
}

// Applies the epilogue in place on the forward's output (the shapes whose state
// pass does not fuse it).
cudaError_t out_gate_after(const gdr_shape* s, const gdr_out_gate* gate, void* y,
                           cudaStream_t st_) {
  return gdr::launch_rmsnorm_gate(y, gate->z, gate->weight, gate->eps, y,
                                  static_cast<long long>(s->B) * s->T * s->H, s->dv,
                                  s->dtype == GDR_F32, st_);
}

gdr_status chunk_fwd_impl(const gdr_shape* shape, int segments, const void* q, const void* k,
                          const void* v, const float* g, const float* beta, const float* lam,
                          const void* b, const void* w, const float* h0, void* o, float* hT,
                          void* workspace, size_t ws_bytes, gdr_stream_t stream,
                          const gdr_out_gate* gate = nullptr) {
  gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  st = check_gates(shape, q, k, v, g, beta, lam, b, w, o);
  if (st != GDR_OK) return st;
  if (gate && (st = check_out_gate(shape, gate, o)) != GDR_OK) return st;
  if ((h0 && !aligned(h0, 16)) || (hT && !aligned(hT, 16))) return GDR_ERR_INVALID_ARG;
  const bool forced = segments > 0;
  if (forced && segments > 1 && !split_allowed(shape)) return GDR_ERR_UNSUPPORTED;
  if (forced && static_cast<long long>(shape->B) * segments > 65535)
    return GDR_ERR_UNSUPPORTED;   // grid z extent of the split scan
  if (forced && segments > 1 && static_cast<long long>(shape->B) * shape->H > 65535)
    return GDR_ERR_UNSUPPORTED;   // grid y extent of the run combination
  const int P = forced ? segments : default_segments(shape);
  size_t need_min = 0, need_full = 0;
  gdr_chunk_fwd_workspace_min(shape, &need_min);
  need_full = split_allowed(shape) ? split_bytes(shape, P)
                                   : (shape->dtype == GDR_BF16 ? two_kernel_bytes(shape) : 0);
  if (need_min > 0 && (!workspace || ws_bytes < need_min || !aligned(workspace, 16)))
    return GDR_ERR_WORKSPACE;
  if (forced && need_full > 0 && ws_bytes < need_full) return GDR_ERR_WORKSPACE;

  const bool f32 = shape->dtype == GDR_F32;
  // the write strength per value channel: the two-kernel path (bf16, full
  // workspace) or the token-order scan
  if ((shape->flags & GDR_BETA_CHANNEL) &&
      (f32 || !workspace || ws_bytes < two_kernel_bytes(shape) || !aligned(workspace, 16))) {
    cudaError_t err = gdr::launch_value_beta_scan(
        value_beta_args(shape, q, k, v, g, beta, h0, o, hT), shape->dk, shape->dv, f32,
        reinterpret_cast<cudaStream_t>(stream));
    if (err == cudaSuccess && gate)
      err = out_gate_after(shape, gate, o, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  gdr::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.lam = lam; a.b = b; a.w = w;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.B = shape->B; a.T = shape->T; a.H = shape->H; a.dv = shape->dv;
  a.flags = shape->flags; a.scale = shape->scale;
  const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  // the epilogue rides in the state pass where the transposed scan runs
  const bool fused = gate && !f32 && ws_bytes >= two_kernel_bytes(shape) &&
                     gdr::scan_transposed(shape->dk, shape->dv, shape->flags);
  if (fused) {
    a.gz = gate->z;
    a.gw = gate->weight;
    a.geps = gate->eps;
  }
  cudaError_t err;
  if (f32) {
    err = gdr::launch_chunk_fwd_f32(a, shape->dk, st_);
  } else {
    int* status = static_cast<int*>(workspace);
    err = cudaMemsetAsync(status, 0, gdr::kStatusWords * sizeof(int), st_);
    if (err == cudaSuccess) {
      // the two-kernel path without the split when the workspace holds the
      // packets but not the run states
      const int runs_req = ws_bytes >= need_full ? P : 1;
      if (ws_bytes >= two_kernel_bytes(shape)) {
        // two kernels: every chunk's intra-chunk work in parallel, then the state pass
        unsigned char* base = static_cast<unsigned char*>(workspace);
        unsigned char* packets = base + gdr::kChunkWorkspaceBytes;
        err = gdr::launch_chunk_prep(a, shape->dk, packets, status, st_);
        if (err == cudaSuccess && runs_req <= 1) {
          err = gdr::launch_chunk_scan(a, shape->dk, packets, status, st_);
        } else if (err == cudaSuccess) {
          // split: each run's local end state H_p (from zero) and transition M_p,
          // then the start states S_p, then every run from its start state
          int runs = 1, seg_chunks = 1;
          split_geometry(shape, runs_req, &runs, &seg_chunks);
          const size_t nrun = static_cast<size_t>(shape->B) * shape->H * runs_req;
          const size_t st_b = nrun * shape->dk * shape->dv * sizeof(float);
          const size_t tr_b = nrun * shape->dk * shape->dk * sizeof(float);
          float* Hl = reinterpret_cast<float*>(base + align256(two_kernel_bytes(shape)));
          float* M = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(Hl) + align256(st_b));
          float* S0 = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(M) + align256(tr_b));
          gdr::ChunkArgs a1 = a;
          a1.h0 = nullptr;
          a1.o = nullptr;
          a1.hT = Hl;
          gdr::ScanSegments s1;
          s1.segments = runs;
          s1.seg_chunks = seg_chunks;
          s1.hT_per_seg = true;
          s1.hT_hom = M;
          err = gdr::launch_chunk_scan(a1, shape->dk, packets, status, st_, s1);
          if (err == cudaSuccess)
            err = gdr::launch_segment_combine(M, Hl, h0, S0, shape->B, shape->H, runs, shape->dk,
                                              shape->dv, st_);
          if (err == cudaSuccess) {
            gdr::ChunkArgs a3 = a;
            a3.h0 = S0;
            gdr::ScanSegments s3;
            s3.segments = runs;
            s3.seg_chunks = seg_chunks;
            s3.h0_per_seg = true;
            err = gdr::launch_chunk_scan(a3, shape->dk, packets, status, st_, s3);
          }
        }
      } else if (gdr::chunk_fwd_pipe_supports(shape->flags)) {
        CUtensorMap tq, tk, tv;
        if (!gdr::make_bthd_tmap(&tq, q, shape->B, shape->T, shape->H, shape->dk) ||
            !gdr::make_bthd_tmap(&tk, k, shape->B, shape->T, shape->H, shape->dk) ||
            !gdr::make_bthd_tmap(&tv, v, shape->B, shape->T, shape->H, shape->dv))
          return GDR_ERR_CUDA;
        err = gdr::launch_chunk_fwd_pipe(a, shape->dk, tq, tk, tv, status, st_);
      } else {
        err = gdr::launch_chunk_fwd_tc(a, shape->dk, status, st_);
      }
    }
  }
  if (err == cudaSuccess && gate && !fused) err = out_gate_after(shape, gate, o, st_);
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

// ---- pipelined two-kernel path: time segments, preparation of segment s + 1
// on `stream` while the scan of segment s runs on `aux` ----
constexpr int kPipePerCta = 1;          // chunks a preparation CTA claims at most
constexpr int kPipeMaxSegments = 64;
constexpr int kPipeTargetSegments = 8;  // segments the default policy aims for
constexpr int kPipeMinChunks = 32;      // chunks per segment, at least

// The segments of a request of S, every one non-empty: up to three segments
// shrink in length by 5/8 from each to the next (the first preparation runs
// alone on every SM and the last state pass alone, so the first is the long
// one; measured 4-7% faster than equal halves or thirds at B * H = 64), more
// are equal. Returns the number used; starts and sizes receive the layout.
int pipe_plan(const gdr_shape* s, int S, int* starts, int* sizes) {
  const int nc = n_chunks_of(s);
  if (S > nc) S = nc;
  if (S <= 3) {
    const double w[3] = {1.0, 0.625, 0.390625};
    double tot = 0.0;
    for (int i = 0; i < S; ++i) tot += w[i];
    int left = nc;
    for (int i = 0; i < S; ++i) {
      const int rest = S - 1 - i;   // segments after this one, one chunk each at least
      int n = i == S - 1 ? left : static_cast<int>(nc * w[i] / tot + 0.5);
      n = std::max(1, std::min(n, left - rest));
      sizes[i] = n;
      left -= n;
    }
  } else {
    const int per = (nc + S - 1) / S;
    S = (nc + per - 1) / per;
    for (int i = 0; i < S; ++i) sizes[i] = std::min(per, nc - i * per);
  }
  for (int i = 0, acc = 0; i < S; ++i) {
    starts[i] = acc;
    acc += sizes[i];
  }
  return S;
}

// status words and packets, then the state handed between segments
// ([B, H, d_k, d_v] fp32) and one work counter per segment
size_t pipelined_bytes(const gdr_shape* s, int S) {
  const size_t st = static_cast<size_t>(s->B) * s->H * s->dk * s->dv * sizeof(float);
  return align256(two_kernel_bytes(s)) + align256(st) + align256(static_cast<size_t>(S) * sizeof(int));
}

gdr_status chunk_fwd_pipelined_impl(const gdr_shape* shape, int segments, const void* q,
                                    const void* k, const void* v, const float* g,
                                    const float* beta, const float* lam, const void* b,
                                    const void* w, const float* h0, void* o, float* hT,
                                    void* workspace, size_t ws_bytes, gdr_stream_t stream,
                                    gdr_stream_t aux_stream, const gdr_out_gate* gate = nullptr) {
  if (segments < 1 || segments > kPipeMaxSegments) return GDR_ERR_INVALID_ARG;
  gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  st = check_gates(shape, q, k, v, g, beta, lam, b, w, o);
  if (st != GDR_OK) return st;
  if (gate && (st = check_out_gate(shape, gate, o)) != GDR_OK) return st;
  if ((h0 && !aligned(h0, 16)) || (hT && !aligned(hT, 16))) return GDR_ERR_INVALID_ARG;
  if (shape->dtype != GDR_BF16) return GDR_ERR_UNSUPPORTED;
  if (!workspace || !aligned(workspace, 16) || ws_bytes < pipelined_bytes(shape, segments))
    return GDR_ERR_WORKSPACE;
  int starts[kPipeMaxSegments], sizes[kPipeMaxSegments];
  const int S = pipe_plan(shape, segments, starts, sizes);

  gdr::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.lam = lam; a.b = b; a.w = w;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.B = shape->B; a.T = shape->T; a.H = shape->H; a.dv = shape->dv;
  a.flags = shape->flags; a.scale = shape->scale;
  const bool fused = gate && gdr::scan_transposed(shape->dk, shape->dv, shape->flags);
  if (fused) {
    a.gz = gate->z;
    a.gw = gate->weight;
    a.geps = gate->eps;
  }
  const cudaStream_t main_ = reinterpret_cast<cudaStream_t>(stream);
  const cudaStream_t aux_ = reinterpret_cast<cudaStream_t>(aux_stream);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  int* status = reinterpret_cast<int*>(base);
  unsigned char* packets = base + gdr::kChunkWorkspaceBytes;
  float* hbuf = reinterpret_cast<float*>(base + align256(two_kernel_bytes(shape)));
  int* counters = reinterpret_cast<int*>(
      reinterpret_cast<unsigned char*>(hbuf) +
      align256(static_cast<size_t>(shape->B) * shape->H * shape->dk * shape->dv * sizeof(float)));

  cudaError_t err = cudaMemsetAsync(status, 0, gdr::kStatusWords * sizeof(int), main_);
  if (err == cudaSuccess) err = cudaMemsetAsync(counters, 0, S * sizeof(int), main_);
  if (err != cudaSuccess) return GDR_ERR_CUDA;
  if (S == 1) {
    err = gdr::launch_chunk_prep(a, shape->dk, packets, status, main_);
    if (err == cudaSuccess) err = gdr::launch_chunk_scan(a, shape->dk, packets, status, main_);
    if (err == cudaSuccess && gate && !fused) err = out_gate_after(shape, gate, o, main_);
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  // one event per segment (its packets are written) and one for the last scan
  cudaEvent_t ev[kPipeMaxSegments + 1];
  int made = 0;
  for (; made <= S; ++made)
    if ((err = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming)) != cudaSuccess) break;
  for (int s = 0; err == cudaSuccess && s < S; ++s) {
    gdr::PrepRange rg;
    rg.chunk0 = starts[s];
    rg.chunks = sizes[s];
    rg.counter = counters + s;
    rg.per_cta = kPipePerCta;
    err = gdr::launch_chunk_prep(a, shape->dk, packets, status, main_, rg);
    if (err == cudaSuccess) err = cudaEventRecord(ev[s], main_);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(aux_, ev[s], 0);
    if (err == cudaSuccess) {
      // segment s starts from h0 or the state segment s - 1 left in hbuf and
      // leaves its end state in hbuf, the last one in hT
      gdr::ChunkArgs as = a;
      as.h0 = s == 0 ? h0 : hbuf;
      as.hT = s == S - 1 ? hT : hbuf;
      gdr::ScanSegments sg;
      sg.chunk0 = rg.chunk0;
      sg.seg_chunks = rg.chunks;
      err = gdr::launch_chunk_scan(as, shape->dk, packets, status, aux_, sg);
    }
  }
  // `stream` resumes after the last scan
  if (err == cudaSuccess) err = cudaEventRecord(ev[S], aux_);
  if (err == cudaSuccess) err = cudaStreamWaitEvent(main_, ev[S], 0);
  if (err == cudaSuccess && gate && !fused) err = out_gate_after(shape, gate, o, main_);
  for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);   // released once completed
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // namespace

extern "C" {

gdr_status gdr_chunk_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, void* o, float* hT, void* workspace,
                         size_t ws_bytes, gdr_stream_t stream) {
  return chunk_fwd_impl(shape, 0, q, k, v, g, beta, lam, b, w, h0, o, hT, workspace, ws_bytes,
                        stream);
}

gdr_status gdr_chunk_fwd_split(const gdr_shape* shape, int segments, const void* q,
                               const void* k, const void* v, const float* g, const float* beta,
                               const float* lam, const void* b, const void* w, const float* h0,
                               void* o, float* hT, void* workspace, size_t ws_bytes,
                               gdr_stream_t stream) {
  if (segments < 1) return GDR_ERR_INVALID_ARG;
  return chunk_fwd_impl(shape, segments, q, k, v, g, beta, lam, b, w, h0, o, hT, workspace,
                        ws_bytes, stream);
}

gdr_status gdr_chunk_fwd_workspace_pipelined(const gdr_shape* shape, int segments,
                                             size_t* bytes) {
  if (!bytes || segments < 1 || segments > kPipeMaxSegments) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  if (shape->dtype != GDR_BF16) return GDR_ERR_UNSUPPORTED;
  *bytes = pipelined_bytes(shape, segments);
  return GDR_OK;
}

gdr_status gdr_chunk_fwd_pipeline_segments(const gdr_shape* shape, int* segments) {
  if (!segments) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  *segments = 1;
  if (shape->dtype != GDR_BF16 || default_segments(shape) > 1) return GDR_OK;
  // the scan CTAs (one per (batch, head), or per (batch, head, 64 value columns)
  // outside the transposed scan) leave at least half of the SMs to the
  // preparation, and the segments average 32 chunks at least: eight equal
  // segments when the scan takes at most a quarter of the SMs, else up to
  // three shrinking ones (measured: at B * H = 64 they beat four and eight)
  const bool tr = gdr::scan_transposed(shape->dk, shape->dv, shape->flags);
  const long long scan_ctas =
      static_cast<long long>(shape->B) * shape->H * (tr ? 1 : shape->dv / 64);
  const int nc = n_chunks_of(shape);
  if (2 * scan_ctas > kSplitTargetCtas) return GDR_OK;
  int S = 1;
  if (4 * scan_ctas <= kSplitTargetCtas) {
    while (S < kPipeTargetSegments && 2 * S * kPipeMinChunks <= nc) S *= 2;
  } else {
    S = std::max(1, std::min(3, nc / kPipeMinChunks));
  }
  *segments = S;
  return GDR_OK;
}

gdr_status gdr_chunk_fwd_pipelined(const gdr_shape* shape, int segments, const void* q,
                                   const void* k, const void* v, const float* g,
                                   const float* beta, const float* lam, const void* b,
                                   const void* w, const float* h0, void* o, float* hT,
                                   void* workspace, size_t ws_bytes, gdr_stream_t stream,
                                   gdr_stream_t aux_stream) {
  return chunk_fwd_pipelined_impl(shape, segments, q, k, v, g, beta, lam, b, w, h0, o, hT,
                                  workspace, ws_bytes, stream, aux_stream);
}

gdr_status gdr_token_fwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, void* o, float* hT,
                         gdr_stream_t stream) {
  gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  st = check_gates(shape, q, k, v, g, beta, lam, b, w, o);
  if (st != GDR_OK) return st;
  if ((h0 && !aligned(h0, 16)) || (hT && !aligned(hT, 16))) return GDR_ERR_INVALID_ARG;
  const bool f32 = shape->dtype == GDR_F32;
  const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  if (shape->flags & GDR_BETA_CHANNEL) {   // its own token-order scan
    const cudaError_t err = gdr::launch_value_beta_scan(
        value_beta_args(shape, q, k, v, g, beta, h0, o, hT), shape->dk, shape->dv, f32, st_);
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  if (shape->B > 65535 || shape->H > 65535) return GDR_ERR_UNSUPPORTED;
  gdr::ChunkArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.lam = lam; a.b = b; a.w = w;
  a.h0 = h0; a.o = o; a.hT = hT;
  a.B = shape->B; a.T = shape->T; a.H = shape->H; a.dv = shape->dv;
  a.flags = shape->flags; a.scale = shape->scale;
  const cudaError_t err = gdr::launch_token_scan(a, shape->dk, f32, st_);
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_chunk_fwd_gated(const gdr_shape* shape, const void* q, const void* k,
                               const void* v, const float* g, const float* beta,
                               const float* lam, const void* b, const void* w, const float* h0,
                               const gdr_out_gate* gate, void* y, float* hT, void* workspace,
                               size_t ws_bytes, gdr_stream_t stream) {
  if (!gate) return GDR_ERR_INVALID_ARG;
  return chunk_fwd_impl(shape, 0, q, k, v, g, beta, lam, b, w, h0, y, hT, workspace, ws_bytes,
                        stream, gate);
}

gdr_status gdr_chunk_fwd_gated_pipelined(const gdr_shape* shape, int segments, const void* q,
                                         const void* k, const void* v, const float* g,
                                         const float* beta, const float* lam, const void* b,
                                         const void* w, const float* h0,
                                         const gdr_out_gate* gate, void* y, float* hT,
                                         void* workspace, size_t ws_bytes, gdr_stream_t stream,
                                         gdr_stream_t aux_stream) {
  if (!gate) return GDR_ERR_INVALID_ARG;
  return chunk_fwd_pipelined_impl(shape, segments, q, k, v, g, beta, lam, b, w, h0, y, hT,
                                  workspace, ws_bytes, stream, aux_stream, gate);
}

gdr_status gdr_chunk_bwd_workspace(const gdr_shape* shape, size_t* bytes) {
  if (!bytes) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  if (shape->flags & GDR_BETA_CHANNEL) {   // the token-order backward (value_beta_bwd.cu)
    *bytes = gdr::value_beta_bwd_workspace_bytes(shape->B, shape->T, shape->H, shape->dk,
                                                 shape->dv);
    return GDR_OK;
  }
  *bytes = gdr::chunk_bwd_workspace_bytes(shape->B, shape->T, shape->H, shape->dk, shape->dv);
  return GDR_OK;
}

static gdr_status bwd_impl(bool token, const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, const void* dO, const float* dhT,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlam,
                         float* db, float* dw, float* dh0, void* workspace, size_t ws_bytes,
                         gdr_stream_t stream) {
  gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  st = check_gates(shape, q, k, v, g, beta, lam, b, w, dO);   // dO takes o's rules
  if (st != GDR_OK) return st;
  const unsigned f = shape->flags;
  const bool need_beta = !((f & GDR_ERASE_CHANNEL) && (f & GDR_WRITE_CHANNEL));
  if (!dq || !dk || !dv || !dg || (need_beta && !dbeta) || ((f & GDR_QMIX) && !dlam) ||
      ((f & GDR_ERASE_CHANNEL) && !db) || ((f & GDR_WRITE_CHANNEL) && !dw))
    return GDR_ERR_INVALID_ARG;
  for (const void* ptr : {static_cast<const void*>(h0), static_cast<const void*>(dhT),
                          static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv), static_cast<const void*>(dg),
                          static_cast<const void*>(dbeta), static_cast<const void*>(dlam),
                          static_cast<const void*>(db), static_cast<const void*>(dw),
                          static_cast<const void*>(dh0)})
    if (ptr && !aligned(ptr, 4)) return GDR_ERR_INVALID_ARG;
  size_t need = 0;
  if (token) {
    gdr_token_bwd_workspace(shape, &need);
  } else {
    gdr_chunk_bwd_workspace(shape, &need);
  }
  if (!workspace || ws_bytes < need || !aligned(workspace, 16)) return GDR_ERR_WORKSPACE;
  if (f & GDR_BETA_CHANNEL) {
    // the write strength per value channel: the token-order backward with
    // chunk checkpoints; no range limit, so the status words stay clear
    gdr::ValueBetaBwdArgs a;
    a.q = q; a.k = k; a.v = v; a.dO = dO; a.g = g; a.beta = beta; a.h0 = h0; a.dhT = dhT;
    a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = dh0;
    a.workspace = workspace;
    a.B = shape->B; a.T = shape->T; a.H = shape->H; a.nk = shape->dk; a.nv = shape->dv;
    a.scale = shape->scale;
    const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t err = cudaMemsetAsync(workspace, 0, gdr::kStatusWords * sizeof(int), st_);
    if (err == cudaSuccess) err = gdr::launch_value_beta_bwd(a, shape->dtype == GDR_F32, st_);
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  gdr::ChunkBwdArgs a;
  a.q = q; a.k = k; a.v = v; a.dO = dO; a.g = g; a.beta = beta; a.lam = lam; a.b = b; a.w = w;
  a.h0 = h0; a.dhT = dhT;
  a.dq = dq; a.dk = dk; a.dv = dv; a.dg = dg; a.dbeta = need_beta ? dbeta : nullptr;
  a.dlam = dlam; a.db = db; a.dw = dw; a.dh0 = dh0; a.workspace = workspace;
  a.B = shape->B; a.T = shape->T; a.H = shape->H; a.dk_dim = shape->dk; a.dv_dim = shape->dv;
  a.flags = f; a.scale = shape->scale;
  const cudaStream_t st_ = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (token) {   // the token-order backward: no range limit, the status words stay clear
    err = cudaMemsetAsync(workspace, 0, gdr::kStatusWords * sizeof(int), st_);
    if (err == cudaSuccess) err = gdr::launch_token_bwd(a, shape->dtype == GDR_F32, st_);
  } else {
    err = gdr::launch_chunk_bwd(a, shape->dtype == GDR_F32, st_);
  }
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_chunk_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, const void* dO, const float* dhT,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlam,
                         float* db, float* dw, float* dh0, void* workspace, size_t ws_bytes,
                         gdr_stream_t stream) {
  return bwd_impl(false, shape, q, k, v, g, beta, lam, b, w, h0, dO, dhT, dq, dk, dv, dg, dbeta,
                  dlam, db, dw, dh0, workspace, ws_bytes, stream);
}

gdr_status gdr_token_bwd_workspace(const gdr_shape* shape, size_t* bytes) {
  if (!bytes) return GDR_ERR_INVALID_ARG;
  const gdr_status st = check_shape(shape, false);
  if (st != GDR_OK) return st;
  *bytes = (shape->flags & GDR_BETA_CHANNEL)
               ? gdr::value_beta_bwd_workspace_bytes(shape->B, shape->T, shape->H, shape->dk,
                                                     shape->dv)
               : gdr::token_bwd_workspace_bytes(shape->B, shape->T, shape->H, shape->dk,
                                                shape->dv);
  return GDR_OK;
}

gdr_status gdr_token_bwd(const gdr_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* lam, const void* b,
                         const void* w, const float* h0, const void* dO, const float* dhT,
                         float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dlam,
                         float* db, float* dw, float* dh0, void* workspace, size_t ws_bytes,
                         gdr_stream_t stream) {
  return bwd_impl(true, shape, q, k, v, g, beta, lam, b, w, h0, dO, dhT, dq, dk, dv, dg, dbeta,
                  dlam, db, dw, dh0, workspace, ws_bytes, stream);
}

gdr_status gdr_chunk_fwd_check(const void* workspace, gdr_stream_t stream, int* detail) {
  return read_status(workspace, stream, detail);
}

gdr_status gdr_chunk_bwd_check(const void* workspace, gdr_stream_t stream, int* detail) {
  return read_status(workspace, stream, detail);
}

gdr_status gdr_recurrent_step(const gdr_shape* shape, const void* q, const void* k,
                              const void* v, const float* g, const float* beta,
                              const float* lam, const void* b, const void* w, float* state,
                              void* o, gdr_stream_t stream) {
  gdr_status st = check_shape(shape, true);
  if (st != GDR_OK) return st;
  st = check_gates(shape, q, k, v, g, beta, lam, b, w, o);
  if (st != GDR_OK) return st;
  if (!state || !aligned(state, 16)) return GDR_ERR_INVALID_ARG;
  if (shape->flags & GDR_BETA_CHANNEL) {   // one token of the token-order scan, in place
    const cudaError_t err = gdr::launch_value_beta_scan(
        value_beta_args(shape, q, k, v, g, beta, state, o, state), shape->dk, shape->dv,
        shape->dtype == GDR_F32, reinterpret_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
  }
  const long long blocks = static_cast<long long>(shape->B) * shape->H;
  if (blocks > 2147483647LL) return GDR_ERR_UNSUPPORTED;
  gdr::StepArgs a;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.lam = lam; a.b = b; a.w = w;
  a.state = state; a.o = o; a.N = shape->B; a.H = shape->H;
  a.flags = shape->flags; a.scale = shape->scale;
  const cudaError_t err = gdr::launch_recurrent_step(a, shape->dk, shape->dv,
                                                     shape->dtype == GDR_F32,
                                                     reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_gate_cumsum(int B, int T, int X, int chunk, const float* g, float* G,
                           gdr_stream_t stream) {
  if (B < 1 || T < 1 || X < 1 || !g || !G) return GDR_ERR_INVALID_ARG;
  if (!aligned(g, 4) || !aligned(G, 4)) return GDR_ERR_INVALID_ARG;
  if (chunk != gdr::kChunkLen) return GDR_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * T * X > kMaxElems * 2LL) return GDR_ERR_UNSUPPORTED;
  if (B > 65535) return GDR_ERR_UNSUPPORTED;
  const cudaError_t err =
      gdr::launch_gate_cumsum(g, G, B, T, X, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

gdr_status gdr_rmsnorm_gate(long long rows, int dv, gdr_dtype dtype, const void* o,
                            const void* z, const float* weight, float eps, void* y,
                            gdr_stream_t stream) {
  if (rows < 0 || dv < 1) return GDR_ERR_INVALID_ARG;
  if (dtype != GDR_F32 && dtype != GDR_BF16) return GDR_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return GDR_ERR_INVALID_ARG;
  if (dv != 64 && dv != 128 && dv != 256) return GDR_ERR_UNSUPPORTED;
  if (rows > (1LL << 40)) return GDR_ERR_UNSUPPORTED;
  if (rows == 0) return GDR_OK;
  if (!o || !z || !weight || !y) return GDR_ERR_INVALID_ARG;
  if (!aligned(o, 16) || !aligned(z, 16) || !aligned(weight, 16) || !aligned(y, 16))
    return GDR_ERR_INVALID_ARG;
  // y is o itself, z itself, or apart from both
  const uintptr_t bytes = static_cast<uintptr_t>(rows) * dv * (dtype == GDR_F32 ? 4 : 2);
  const uintptr_t py = reinterpret_cast<uintptr_t>(y);
  for (const void* src : {o, z}) {
    const uintptr_t ps = reinterpret_cast<uintptr_t>(src);
    if (ps != py && ps < py + bytes && py < ps + bytes) return GDR_ERR_INVALID_ARG;
  }
  const cudaError_t err = gdr::launch_rmsnorm_gate(o, z, weight, eps, y, rows, dv,
                                                   dtype == GDR_F32,
                                                   reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDR_OK : GDR_ERR_CUDA;
}

}  // extern "C"
