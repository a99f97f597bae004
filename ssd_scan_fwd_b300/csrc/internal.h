// internal.h -- shared declarations of the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <cstdint>

#include "ssd.h"

namespace ssd {

// A validated problem: sizes, chunking and device pointers of one call.
struct Problem {
  int64_t B, L, H, P, G, N;
  int io;      // ssd_dtype
  int64_t Q_req;  // chunk length the caller asked for (0 = library default)
  int64_t Q;   // chunk length of the chunked path
  int64_t nc;  // ceil(L / Q)
  const void* x;
  const float* dt;
  const float* A;
  const void* Bm;
  const void* Cm;
  const float* D;
  const float* init;
  void* y;
  float* final_state;
  // steps around the scan (ssd_fwd_ex): Δ = softplus?(dt + dt_bias), y ← y · silu(z)
  const float* dt_bias = nullptr;
  int dt_softplus = 0;
  const void* z = nullptr;
  // complex decay (ssd_fwd_rot): rotation angles [B,L,H] and the imaginary
  // parts of the initial / final states [B,H,P,N]
  const float* theta = nullptr;
  const float* init_im = nullptr;
  float* final_im = nullptr;
  bool complex_decay = false;  // set by the complex-decay entry points (theta may be null in size queries)
  // status word: the tensor-core kernels of the chunked path write
  // SSD_ERR_TIMEOUT here when one of their bounded waits gives up (null: not recorded)
  int32_t* err = nullptr;
  // retrieval rank (ssd_fwd_mimo, fused path only): L counts rows = tokens ×
  // 2^rank_log2, the R rows of a token consecutive; dt has Ltok = L >> rank_log2
  // tokens per batch row
  int rank_log2 = 0;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---- chunked path (chunked.cu): four kernels; chunk states and outputs go ----
// ---- to the tensor-core kernels where state_tc.cu / scan_tc.cu apply      ----
// phi: in-chunk sums of p.theta (written only when p.theta is set).
cudaError_t launch_chunk_cumsum(const Problem& p, float* dA_cs, float* dt_c, cudaStream_t s,
                                float* phi = nullptr);
cudaError_t launch_chunk_state(const Problem& p, const float* dA_cs, const float* dt_c,
                               float* states, cudaStream_t s);
// states_bf (optional): write the states entering each chunk as bf16 there
// ([B][nc][H][P][N]) instead of fp32 over `states`.
cudaError_t launch_state_passing(const Problem& p, const float* dA_cs, float* states,
                                 cudaStream_t s, void* states_bf = nullptr);
// The forward pass with the complex decay (chunked path): cumsum
// of Δ·A and θ, real and imaginary chunk states, the complex state
// recurrence (writes p.final_state / p.final_im), the chunk outputs.
// Workspace: dA_cs, dt_c, phi [B][H][nc][Q], st_re, st_im [B][nc][H][P][N].
// With re_bf, im_bf (bf16 [B][nc][H][P][N], where scan_tc_supported(p)) the
// recurrence writes the entering states there and the chunk outputs come
// from the tensor-core kernel of scan_tc.cu.
cudaError_t launch_rot(const Problem& p, float* dA_cs, float* dt_c, float* phi, float* st_re, float* st_im,
                       cudaStream_t s, void* re_bf = nullptr, void* im_bf = nullptr);

// ---- chunk outputs on the tensor cores (scan_tc.cu) ----
// bf16 io, headdim 64, dstate 16, 64, 128 or 256, chunk 128 (SSD_CHUNK_SCAN_CUDA_CORES=1
// turns it off).  re_bf, im_bf: bf16 states entering each chunk,
// [B][nc][H][P][N]; phi (complex decay) null for the real method.
bool scan_tc_supported(const Problem& p);
cudaError_t launch_chunk_scan_tc(const Problem& p, const float* dA_cs, const float* dt_c, const float* phi,
                                 const void* re_bf, const void* im_bf, cudaStream_t s);

// Adjoint chunk states of the backward pass, Σ_i exp(cs_i) dy_i C_iᵀ per
// chunk (same layout as the chunk states).
cudaError_t launch_chunk_state_adjoint(const Problem& p, const void* dy, const float* dA_cs,
                                       float* gstates, cudaStream_t s);
cudaError_t launch_chunk_scan(const Problem& p, const float* dA_cs, const float* dt_c,
                              const float* states, cudaStream_t s);

// ---- fused path (fused.cu): one persistent tcgen05 kernel ----
bool fused_supported(const Problem& p);  // bf16, headdim 64, dstate 16, 64 or 128, chunk 128
bool fused_preferred(const Problem& p);  // supported, and the better path for SSD_ALGO_AUTO
// Workspace bytes the fused kernel uses for p when it may use at most
// `max_bytes` (the plan shrinks its sequence segmentation to fit; 256 bytes
// always suffice).  launch_fused must be given the same `max_bytes`.
size_t fused_workspace_bytes(const Problem& p, size_t max_bytes = SIZE_MAX);
cudaError_t launch_fused(const Problem& p, void* workspace, cudaStream_t s, size_t max_bytes = SIZE_MAX);
// The backward pass's recomputed states, on the fused path's states kernel
// (bf16, P = 64, N = 128, chunk 128): the state entering every chunk (hin)
// and the adjoint leaving every chunk (gout), both bf16 [B][nc][H][P][N],
// and dinit (fp32, if non-null) from dfinal (or zero).  Timeouts go to *err.
// The walks are cut into one contiguous range of steps per CTA, handing the
// state over at each cut: `flags` (states_walks(p) · 2 words, zero on entry)
// and `slots` (states_walks(p) · 2 · P · N fp32).
bool states_hin_supported(const Problem& p);
int states_walks(const Problem& p);
cudaError_t launch_states_walks(const Problem& p, void* hin, const void* dy, const float* dfinal, float* dinit,
                                void* gout, uint32_t* flags, float* slots, int32_t* err, cudaStream_t s);

// A 3-D tensor map over a bf16 [B][L][W] array (fused.cu): boxes of 64
// columns (128-byte swizzle) by box_rows rows.
bool make_tma_map_bf16(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t W, int box_rows);
// A 4-D tensor map over an fp32 [B][L][G][N] array (fused.cu): boxes of 32
// columns (128-byte swizzle) by box_rows tokens of one group and batch row;
// coordinates (n, g, t, b), rows past L clipped.
bool make_tma_map_f32_bltgn(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t G, int64_t N,
                            int box_rows);
// A 4-D tensor map over a bf16 [B][L][G][N] array with N < 64: boxes of 64
// columns (the columns past N read as zero) by box_rows tokens of one group
// and batch row, 128-byte swizzle; coordinates (0, g, t, b).
bool make_tma_map_bf16_narrow(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t G, int64_t N,
                              int box_rows);

// ---- chunk states on the tensor cores (state_tc.cu) ----
// S[b][c][h][p][n] = Σ_i w_i xin_i[p] bin_i[n] for bf16 io, P = 64, N = 16,
// 64, 128 or 256, chunk 64 or 128; the weights by mode as in chunk_state_kernel (0 forward, 1
// adjoint, 2 / 3 real / imaginary rotation).  Returns cudaErrorNotSupported
// for any other shape (the caller then uses the CUDA-core kernel).
bool chunk_state_tc_supported(const Problem& p);
cudaError_t launch_chunk_state_tc(const Problem& p, int mode, const void* xin, const void* bin,
                                  const float* dA_cs, const float* dt_c, const float* phi, float* states,
                                  cudaStream_t s);

// ---- recurrent step (step.cu) ----
struct StepProblem {
  int64_t B, H, P, G, N;
  int io;  // ssd_dtype
  const void* x;
  const float* dt;
  const float* A;
  const void* Bm;
  const void* Cm;
  const float* D;
  float* state;
  void* y;
};
cudaError_t launch_step(const StepProblem& q, cudaStream_t s);

// ---- gradient (bwd.cu) ----
// fwd: the forward problem (Q = bwd_chunk(...); y and final_state unused).
struct BwdProblem {
  Problem fwd;
  const void* dy;       // [B,L,H,P] io dtype
  const float* dfinal;  // [B,H,P,N] or null
  void* dx;             // [B,L,H,P] io dtype
  float* ddt;           // [B,L,H]
  float* dA;            // [H]
  void* dBm;            // [B,L,G,N] io dtype
  void* dCm;            // [B,L,G,N] io dtype
  float* dD;            // [H] or null
  float* dinit;         // [B,H,P,N] or null
};
struct BwdWs {
  size_t off_cs, off_dt, off_states, off_gstates, off_db, off_dc, off_wflag, off_wslot, total;
};
BwdWs bwd_ws(const Problem& p);
// The backward pass's state recurrences run as walks of the states kernel
// (the tensor-core path), so its workspace holds no fp32 per-chunk states.
bool bwd_walks(const Problem& p);
// Chunk length of the backward pass for a requested chunk_size (0: the
// default, 128 on the tensor-core path, else 64); 0 when unsupported.
int bwd_chunk(const Problem& p, int64_t requested);
bool bwd_tc_supported(const Problem& p);  // bf16, headdim 64, dstate 128
// states_bf, gstates_bf: bf16 h_in and Gout per chunk, [B][nc][H][P][N].
cudaError_t launch_bwd_chunk_tc(const BwdProblem& q, const float* dA_cs, const float* dt_c, const void* states_bf,
                                const void* gstates_bf, float* dB_acc, float* dC_acc, cudaStream_t s);
int bwd_max_headdim();  // largest headdim it supports
cudaError_t launch_bwd(const BwdProblem& q, void* workspace, cudaStream_t s);

// Fixed device scratch for the allocation-free entry point (fused.cu).
size_t static_scratch_bytes();
cudaError_t static_scratch_ptr(void** out);

}  // namespace ssd
