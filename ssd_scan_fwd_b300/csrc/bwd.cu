// bwd.cu -- gradient of the SSD forward pass: fp32 CUDA-core arithmetic, io
// fp32 or bf16.
//
// The function differentiated is the recurrence of the page "Mamba-3 深度剖析
// - 02. SSM 基础回顾与演进 (Foundations of SSM)" (§2.1.2: h_t = α_t h_{t-1} +
// Δ_t x_t B_tᵀ, α_t = e^{Δ_t A}, y_t = h_t C_t, plus the skip term D x_t of
// §2.1.1); the scalar is Σ dy ⊙ y + Σ dfinal ⊙ final_state.  As the page
// "从 SSM 的长期记忆问题，到 Mamba 的选择性机制与硬件感知扫描" has it for
// the hardware-aware scan, the backward pass recomputes the states rather than
// reading stored ones: the states entering each chunk are recomputed with the
// chunked forward kernels (chunk_cumsum, chunk_state, state_passing).
//
// With G_t = ∂/∂h_t of the scalar (its whole dependence on h_t), inside chunk c
// (tokens i = 0..Q-1, in-chunk sums cs_i of a = Δ·A, last = Q-1):
//   Gout[c] = G after the chunk's last token, through later chunks only:
//     Gout[nc-1] = dfinal,  Gout[c-1] = e^{cs_last} Gout[c] + dS_c,
//     dS_c = Σ_i e^{cs_i} dy_i C_iᵀ                 (adjoint chunk state)
//   G_t = Σ_{s≥t} e^{cs_s - cs_t} dy_s C_sᵀ + e^{cs_last - cs_t} Gout[c]
//   u_t = G_t B_t,  dx_t = D dy_t + Δ_t u_t
//   dB_t = Δ_t G_tᵀ x_t,  dC_t = h_tᵀ dy_t       (summed over a group's heads)
//   da_t = <G_t, α_t h_{t-1}>                     (a_t = Δ_t A = log α_t)
//   dΔ_t = x_t·u_t + A da_t,  dA = Σ Δ_t da_t,  dD = Σ dy_t·x_t
//   dinit = e^{cs_last} Gout[0] + dS_0 (the G entering chunk 0)
// Every product of G_t or h_t with another operand expands into intra-chunk
// matrices of the same masked form as the forward pass, with the mask
// e^{cs_s - cs_j} (s ≥ j, never positive in the exponent):
//   CB[s][j] = C_s·B_j,  DX[s][j] = dy_s·x_j,
//   u_t      = Σ_{s≥t} e^{cs_s-cs_t} CB[s][t] dy_s + e^{cs_last-cs_t} Gout B_t
//   dB_t     = Δ_t (Σ_{s≥t} e^{cs_s-cs_t} DX[s][t] C_s + e^{cs_last-cs_t} Goutᵀ x_t)
//   dC_s     = Σ_{j≤s} e^{cs_s-cs_j} Δ_j DX[s][j] B_j + e^{cs_s} h_inᵀ dy_s
//   da_t     = Σ_{s≥t} Σ_{j<t} W[s][j] + Σ_{s≥t} e^{cs_s} C_s·(h_inᵀ dy_s)
//              + Σ_{j<t} e^{cs_last-cs_j} Δ_j x_j·(Gout B_j) + e^{cs_last} <Gout, h_in>
//              with W[s][j] = e^{cs_s-cs_j} Δ_j DX[s][j] CB[s][j]
// (α_t h_{t-1} holds the inputs j < t only, so da_t needs no cancellation).

#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"

namespace ssd {
namespace {

constexpr int kQ = 64;    // chunk length of the backward pass
constexpr int kT = 256;   // threads per block
constexpr int kNT = 32;   // state columns per slice
constexpr int kPMax = 128;

__device__ __forceinline__ float ld_f(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_f(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

// ---------------------------------------------------------------------------
// Adjoint chunk states dS_c[p][n] = Σ_i e^{cs_i} dy_i[p] C_i[n].  One block
// per (chunk, head, batch); output [B][nc][H][P][N].
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kT) bwd_dstate_kernel(const T* __restrict__ dy, const T* __restrict__ Cm,
                                                        const float* __restrict__ dA_cs, int64_t L, int64_t H,
                                                        int P, int G, int N, int64_t nc,
                                                        float* __restrict__ gstates) {
  constexpr int TK = 32;
  constexpr int R = 16;
  extern __shared__ float smem[];
  float* ys = smem;           // [TK][P], rows scaled by e^{cs_i}
  float* cs_ = smem + TK * P; // [TK][N]
  __shared__ float w_s[kQ];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (H / G);
  const int tid = threadIdx.x;
  const float* cs = dA_cs + ((b * H + h) * nc + c) * kQ;
  for (int i = tid; i < kQ; i += kT) w_s[i] = expf(cs[i]);
  __syncthreads();
  const int PN = P * N;
  for (int base = 0; base < PN; base += kT * R) {
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int k0 = 0; k0 < kQ; k0 += TK) {
      for (int e = tid; e < TK * P; e += kT) {
        const int k = e / P, p = e - k * P;
        const int64_t t = c * kQ + k0 + k;
        ys[e] = (t < L) ? ld_f(dy, ((b * L + t) * H + h) * P + p) * w_s[k0 + k] : 0.f;
      }
      for (int e = tid; e < TK * N; e += kT) {
        const int k = e / N, n = e - k * N;
        const int64_t t = c * kQ + k0 + k;
        cs_[e] = (t < L) ? ld_f(Cm, ((b * L + t) * G + g) * N + n) : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = base + tid + kT * r;
        if (e < PN) {
          const int p = e / N, n = e - p * N;
          float s = 0.f;
#pragma unroll 8
          for (int k = 0; k < TK; ++k) s = fmaf(ys[k * P + p], cs_[k * N + n], s);
          acc[r] += s;
        }
      }
      __syncthreads();
    }
    float* out = gstates + ((b * nc + c) * H + h) * (int64_t)PN;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int e = base + tid + kT * r;
      if (e < PN) out[e] = acc[r];
    }
  }
}

// ---------------------------------------------------------------------------
// The adjoint recurrence across chunks, last chunk first.  On entry slot c
// holds dS_c; on exit it holds Gout[c], and dinit = the G entering chunk 0.
// One thread per state entry.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kT) bwd_state_passing_kernel(const float* __restrict__ dA_cs,
                                                               const float* __restrict__ dfinal,
                                                               float* __restrict__ gstates,
                                                               float* __restrict__ dinit, int64_t H,
                                                               int64_t PN, int64_t nc) {
  const int64_t e = (int64_t)blockIdx.x * kT + threadIdx.x;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  if (e >= PN) return;
  float gv = dfinal ? dfinal[(b * H + h) * PN + e] : 0.f;
  const float* cs = dA_cs + (b * H + h) * nc * kQ;
  for (int64_t c = nc - 1; c >= 0; --c) {
    float* slot = gstates + ((b * nc + c) * H + h) * PN + e;
    const float ds = *slot;
    *slot = gv;
    gv = fmaf(expf(cs[c * kQ + kQ - 1]), gv, ds);
  }
  if (dinit) dinit[(b * H + h) * PN + e] = gv;
}

// ---------------------------------------------------------------------------
// Gradients of one chunk of one head.  One block per (chunk, head, batch).
// ---------------------------------------------------------------------------
struct ChunkGradArgs {
  const void* x;
  const void* dy;
  const void* Bm;
  const void* Cm;
  const float* A;
  const float* D;
  const float* dA_cs;
  const float* dt_c;
  const float* states;   // h_in per chunk
  const float* gstates;  // Gout per chunk
  void* dx;
  float* ddt;
  float* dB_acc;
  float* dC_acc;
  float* dA;
  float* dD;
  int64_t L, H, nc;
  int P, G, N;
};

constexpr int kLdQ = kQ + 1;

template <int PMAX>
struct ChunkSmem {
  static constexpr int kLdP = PMAX + 1;
  static constexpr int kXs = 0;                         // x  [Q][P+1]
  static constexpr int kDys = kXs + kQ * kLdP;          // dy [Q][P+1]
  static constexpr int kM1 = kDys + kQ * kLdP;          // e^{cs_s-cs_j} CB[s][j]          (j ≤ s)
  static constexpr int kM2 = kM1 + kQ * kLdQ;           // DX, then e^{cs_s-cs_j} DX[s][j] (j ≤ s)
  static constexpr int kM3 = kM2 + kQ * kLdQ;           // e^{cs_s-cs_j} Δ_j DX[s][j]      (j ≤ s)
  static constexpr int kM4 = kM3 + kQ * kLdQ;           // W[s][j] = M3 · CB               (j ≤ s)
  static constexpr int kBs = kM4 + kQ * kLdQ;           // B slice [Q][NT+1]
  static constexpr int kCs = kBs + kQ * (kNT + 1);      // C slice [Q][NT+1]
  static constexpr int kGs = kCs + kQ * (kNT + 1);      // Gout slice [P][NT+1]
  static constexpr int kHs = kGs + PMAX * (kNT + 1);    // h_in slice [P][NT+1]
  static constexpr int kVec = kHs + PMAX * (kNT + 1);   // per-token vectors
  // vectors: cs, dl, xu, gbx, a1, rp (Q+1), red (kT)
  static constexpr int kFloats = kVec + 6 * kQ + 1 + kT;
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

template <typename T, int PMAX>
__global__ void __launch_bounds__(kT) bwd_chunk_kernel(const ChunkGradArgs a) {
  using S = ChunkSmem<PMAX>;
  constexpr int LDP = S::kLdP;
  constexpr int RQQ = kQ * kQ / kT;      // 16 (s, j) entries per thread
  constexpr int RQP = kQ * PMAX / kT;    // (t, p) entries per thread
  extern __shared__ float sm[];
  float* xs = sm + S::kXs;
  float* dys = sm + S::kDys;
  float* M1 = sm + S::kM1;
  float* M2 = sm + S::kM2;
  float* M3 = sm + S::kM3;
  float* M4 = sm + S::kM4;
  float* Bs = sm + S::kBs;
  float* Cs = sm + S::kCs;
  float* Gs = sm + S::kGs;
  float* Hs = sm + S::kHs;
  float* cs = sm + S::kVec;
  float* dl = cs + kQ;
  float* xu = dl + kQ;      // x_t·u_t
  float* gbx = xu + kQ;     // x_t·(Gout B_t)
  float* a1 = gbx + kQ;     // e^{cs_t} C_t·(h_inᵀ dy_t)
  float* rp = a1 + kQ;      // [Q+1]: strict rectangle sums of W
  float* red = rp + kQ + 1; // [kT] block reduction

  const T* x = static_cast<const T*>(a.x);
  const T* dy = static_cast<const T*>(a.dy);
  const T* Bm = static_cast<const T*>(a.Bm);
  const T* Cm = static_cast<const T*>(a.Cm);
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (a.H / a.G);
  const int P = a.P, N = a.N;
  const int tid = threadIdx.x;
  const int64_t t0 = c * kQ;

  for (int i = tid; i < kQ; i += kT) {
    cs[i] = a.dA_cs[((b * a.H + h) * a.nc + c) * kQ + i];
    dl[i] = a.dt_c[((b * a.H + h) * a.nc + c) * kQ + i];
    xu[i] = 0.f;
    gbx[i] = 0.f;
    a1[i] = 0.f;
  }
  for (int e = tid; e < kQ * P; e += kT) {
    const int i = e / P, p = e - i * P;
    const int64_t t = t0 + i;
    const int64_t o = ((b * a.L + t) * a.H + h) * P + p;
    xs[i * LDP + p] = t < a.L ? ld_f(x, o) : 0.f;
    dys[i * LDP + p] = t < a.L ? ld_f(dy, o) : 0.f;
  }
  __syncthreads();
  // DX[s][j] = dy_s · x_j
#pragma unroll
  for (int r = 0; r < RQQ; ++r) {
    const int e = tid + kT * r;
    const int s = e / kQ, j = e - s * kQ;
    float v = 0.f;
    for (int p = 0; p < P; ++p) v = fmaf(dys[s * LDP + p], xs[j * LDP + p], v);
    M2[s * kLdQ + j] = v;
  }
  // CB[s][j] = C_s · B_j and GB[t][p] = Σ_n B_t[n] Gout[p][n], over state slices;
  // γ = <Gout, h_in>
  float cb[RQQ], gb[RQP];
#pragma unroll
  for (int r = 0; r < RQQ; ++r) cb[r] = 0.f;
#pragma unroll
  for (int r = 0; r < RQP; ++r) gb[r] = 0.f;
  float gam = 0.f;
  const float* hin = a.states + ((b * a.nc + c) * a.H + h) * (int64_t)P * N;
  const float* gout = a.gstates + ((b * a.nc + c) * a.H + h) * (int64_t)P * N;
  auto load_slices = [&](int n0) {
    for (int e = tid; e < kQ * kNT; e += kT) {
      const int i = e / kNT, k = e - i * kNT;
      const int64_t t = t0 + i;
      const bool ok = t < a.L && n0 + k < N;
      const int64_t o = ((b * a.L + t) * a.G + g) * N + n0 + k;
      Bs[i * (kNT + 1) + k] = ok ? ld_f(Bm, o) : 0.f;
      Cs[i * (kNT + 1) + k] = ok ? ld_f(Cm, o) : 0.f;
    }
    for (int e = tid; e < P * kNT; e += kT) {
      const int p = e / kNT, k = e - p * kNT;
      const bool ok = n0 + k < N;
      Gs[p * (kNT + 1) + k] = ok ? gout[(int64_t)p * N + n0 + k] : 0.f;
      Hs[p * (kNT + 1) + k] = ok ? hin[(int64_t)p * N + n0 + k] : 0.f;
    }
  };
  for (int n0 = 0; n0 < N; n0 += kNT) {
    __syncthreads();
    load_slices(n0);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < RQQ; ++r) {
      const int e = tid + kT * r;
      const int s = e / kQ, j = e - s * kQ;
      float v = 0.f;
#pragma unroll 8
      for (int k = 0; k < kNT; ++k) v = fmaf(Cs[s * (kNT + 1) + k], Bs[j * (kNT + 1) + k], v);
      cb[r] += v;
    }
#pragma unroll
    for (int r = 0; r < RQP; ++r) {
      const int e = tid + kT * r;
      const int t = e / PMAX, p = e - t * PMAX;
      if (p < P) {
        float v = 0.f;
#pragma unroll 8
        for (int k = 0; k < kNT; ++k) v = fmaf(Bs[t * (kNT + 1) + k], Gs[p * (kNT + 1) + k], v);
        gb[r] += v;
      }
    }
    for (int e = tid; e < P * kNT; e += kT) {
      const int p = e / kNT, k = e - p * kNT;
      gam = fmaf(Gs[p * (kNT + 1) + k], Hs[p * (kNT + 1) + k], gam);
    }
  }
  // Masked matrices.  dD (Σ_t dy_t·x_t) is the trace of DX.
  float ddsum = 0.f;
#pragma unroll
  for (int r = 0; r < RQQ; ++r) {
    const int e = tid + kT * r;
    const int s = e / kQ, j = e - s * kQ;
    const float dxv = M2[s * kLdQ + j];
    if (s == j) ddsum += dxv;
    const bool lower = j <= s;
    const float E = lower ? expf(cs[s] - cs[j]) : 0.f;
    const float wc = E * dl[j] * dxv;
    M1[s * kLdQ + j] = E * cb[r];
    M2[s * kLdQ + j] = E * dxv;
    M3[s * kLdQ + j] = wc;
    M4[s * kLdQ + j] = wc * cb[r];
  }
  __syncthreads();
  const float cs_last = cs[kQ - 1];
  // u_t = Σ_{s≥t} M1[s][t] dy_s + e^{cs_last-cs_t} GB[t];  dx_t = D dy_t + Δ_t u_t
  const float Dh = a.D ? a.D[h] : 0.f;
  T* dxo = static_cast<T*>(a.dx);
#pragma unroll
  for (int r = 0; r < RQP; ++r) {
    const int e = tid + kT * r;
    const int t = e / PMAX, p = e - t * PMAX;
    if (p < P) {
      float v = 0.f;
      for (int s = t; s < kQ; ++s) v = fmaf(M1[s * kLdQ + t], dys[s * LDP + p], v);
      const float eg = expf(cs_last - cs[t]);
      const float u = fmaf(eg, gb[r], v);
      const float xv = xs[t * LDP + p];
      atomicAdd(&xu[t], xv * u);
      atomicAdd(&gbx[t], xv * gb[r]);
      const int64_t tt = t0 + t;
      if (tt < a.L) st_f(dxo, ((b * a.L + tt) * a.H + h) * P + p, fmaf(Dh, dys[t * LDP + p], dl[t] * u));
    }
  }
  // dB and dC over state slices; a1_t = e^{cs_t} C_t·(h_inᵀ dy_t)
  for (int n0 = 0; n0 < N; n0 += kNT) {
    __syncthreads();
    load_slices(n0);
    __syncthreads();
    for (int e = tid; e < kQ * kNT; e += kT) {
      const int t = e / kNT, k = e - t * kNT;
      float xg = 0.f, yh = 0.f;
      for (int p = 0; p < P; ++p) {
        xg = fmaf(xs[t * LDP + p], Gs[p * (kNT + 1) + k], xg);
        yh = fmaf(dys[t * LDP + p], Hs[p * (kNT + 1) + k], yh);
      }
      float vb = 0.f, vc = 0.f;
      for (int s = t; s < kQ; ++s) vb = fmaf(M2[s * kLdQ + t], Cs[s * (kNT + 1) + k], vb);
      for (int j = 0; j <= t; ++j) vc = fmaf(M3[t * kLdQ + j], Bs[j * (kNT + 1) + k], vc);
      const float ecs = expf(cs[t]);
      const float db = dl[t] * fmaf(expf(cs_last - cs[t]), xg, vb);
      const float dc = fmaf(ecs, yh, vc);
      atomicAdd(&a1[t], ecs * Cs[t * (kNT + 1) + k] * yh);
      const int64_t tt = t0 + t;
      if (tt < a.L && n0 + k < N) {
        const int64_t o = ((b * a.L + tt) * a.G + g) * N + n0 + k;
        atomicAdd(a.dB_acc + o, db);
        atomicAdd(a.dC_acc + o, dc);
      }
    }
  }
  // rp[t] = Σ_{s≥t} Σ_{j<t} W[s][j], built from its differences
  // rp[k+1] - rp[k] = Σ_{s>k} W[s][k] - Σ_{j<k} W[k][j]
  for (int k = tid; k < kQ; k += kT) {
    float v = 0.f;
    for (int s = k + 1; s < kQ; ++s) v += M4[s * kLdQ + k];
    for (int j = 0; j < k; ++j) v -= M4[k * kLdQ + j];
    rp[k + 1] = v;
  }
  if (tid == 0) rp[0] = 0.f;
  red[tid] = gam;
  __syncthreads();
  if (tid < 32) {
    float v = 0.f;
    for (int i = tid; i < kT; i += 32) v += red[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tid == 0) {
      // sequential scans over the chunk: prefix of rp, suffix of a1, exclusive prefix of β1
      const float gamma = expf(cs_last) * v;
      float run = 0.f;
      for (int k = 0; k < kQ; ++k) {
        run += rp[k];
        rp[k] = run;
      }
      float suf = 0.f;
      for (int k = kQ - 1; k >= 0; --k) {
        suf += a1[k];
        a1[k] = suf;
      }
      float pre = 0.f, dAsum = 0.f;
      for (int k = 0; k < kQ; ++k) {
        const float da = rp[k] + a1[k] + pre + gamma;
        pre += dl[k] * expf(cs_last - cs[k]) * gbx[k];
        const int64_t tt = t0 + k;
        if (tt < a.L) a.ddt[(b * a.L + tt) * a.H + h] = fmaf(a.A[h], da, xu[k]);
        dAsum = fmaf(dl[k], da, dAsum);
      }
      atomicAdd(a.dA + h, dAsum);
    }
  }
  __syncthreads();
  red[tid] = ddsum;
  __syncthreads();
  if (tid < 32) {
    float v = 0.f;
    for (int i = tid; i < kT; i += 32) v += red[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (tid == 0 && a.dD) atomicAdd(a.dD + h, v);
  }
}

// fp32 group sums -> io dtype
template <typename T>
__global__ void __launch_bounds__(kT) bwd_convert_kernel(const float* __restrict__ src, T* __restrict__ dst,
                                                         int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * kT + threadIdx.x; i < n; i += (int64_t)gridDim.x * kT)
    st_f(dst, i, src[i]);
}

template <typename T, int PMAX>
cudaError_t launch_chunk_grad(const ChunkGradArgs& ga, int64_t B, cudaStream_t s) {
  using Sm = ChunkSmem<PMAX>;
  cudaError_t e = cudaFuncSetAttribute(bwd_chunk_kernel<T, PMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Sm::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)ga.nc, (unsigned)ga.H, (unsigned)B);
  bwd_chunk_kernel<T, PMAX><<<grid, kT, Sm::kBytes, s>>>(ga);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_bwd_t(const BwdProblem& q, const BwdWs& w, char* ws, cudaStream_t s) {
  const Problem& p = q.fwd;
  float* dA_cs = reinterpret_cast<float*>(ws + w.off_cs);
  float* dt_c = reinterpret_cast<float*>(ws + w.off_dt);
  float* states = reinterpret_cast<float*>(ws + w.off_states);
  float* gstates = reinterpret_cast<float*>(ws + w.off_gstates);
  float* dB_acc = reinterpret_cast<float*>(ws + w.off_db);
  float* dC_acc = reinterpret_cast<float*>(ws + w.off_dc);
  const int64_t nbc = p.B * p.L * p.G * p.N;
  cudaError_t e;
  if ((e = cudaMemsetAsync(dB_acc, 0, (size_t)nbc * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dC_acc, 0, (size_t)nbc * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(q.dA, 0, (size_t)p.H * 4, s)) != cudaSuccess) return e;
  if (q.dD && (e = cudaMemsetAsync(q.dD, 0, (size_t)p.H * 4, s)) != cudaSuccess) return e;
  // forward recompute: the state entering each chunk
  if ((e = launch_chunk_cumsum(p, dA_cs, dt_c, s)) != cudaSuccess) return e;
  if ((e = launch_chunk_state(p, dA_cs, dt_c, states, s)) != cudaSuccess) return e;
  if ((e = launch_state_passing(p, dA_cs, states, s)) != cudaSuccess) return e;
  // adjoint chunk states, then the adjoint recurrence (last chunk first)
  {
    const size_t smem = sizeof(float) * 32 * (size_t)(p.P + p.N);
    if ((e = cudaFuncSetAttribute(bwd_dstate_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
    bwd_dstate_kernel<T><<<grid, kT, smem, s>>>((const T*)q.dy, (const T*)p.Cm, dA_cs, p.L, p.H, (int)p.P,
                                                 (int)p.G, (int)p.N, p.nc, gstates);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int64_t PN = p.P * p.N;
    dim3 grid((unsigned)((PN + kT - 1) / kT), (unsigned)p.H, (unsigned)p.B);
    bwd_state_passing_kernel<<<grid, kT, 0, s>>>(dA_cs, q.dfinal, gstates, q.dinit, p.H, PN, p.nc);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  ChunkGradArgs ga;
  ga.x = p.x;
  ga.dy = q.dy;
  ga.Bm = p.Bm;
  ga.Cm = p.Cm;
  ga.A = p.A;
  ga.D = p.D;
  ga.dA_cs = dA_cs;
  ga.dt_c = dt_c;
  ga.states = states;
  ga.gstates = gstates;
  ga.dx = q.dx;
  ga.ddt = q.ddt;
  ga.dB_acc = dB_acc;
  ga.dC_acc = dC_acc;
  ga.dA = q.dA;
  ga.dD = q.dD;
  ga.L = p.L;
  ga.H = p.H;
  ga.nc = p.nc;
  ga.P = (int)p.P;
  ga.G = (int)p.G;
  ga.N = (int)p.N;
  e = p.P <= 64 ? launch_chunk_grad<T, 64>(ga, p.B, s) : launch_chunk_grad<T, 128>(ga, p.B, s);
  if (e != cudaSuccess) return e;
  const unsigned cgrid = (unsigned)std::min<int64_t>((nbc + kT - 1) / kT, 4096);
  bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dB_acc, (T*)q.dBm, nbc);
  bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dC_acc, (T*)q.dCm, nbc);
  return cudaGetLastError();
}

}  // namespace

BwdWs bwd_ws(const Problem& p) {
  BwdWs w;
  const size_t ncs = align_up((size_t)(p.B * p.H * p.nc * p.Q) * 4, 256);
  const size_t nst = align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 4, 256);
  const size_t nbc = align_up((size_t)(p.B * p.L * p.G * p.N) * 4, 256);
  w.off_cs = 0;
  w.off_dt = ncs;
  w.off_states = 2 * ncs;
  w.off_gstates = w.off_states + nst;
  w.off_db = w.off_gstates + nst;
  w.off_dc = w.off_db + nbc;
  w.total = w.off_dc + nbc;
  return w;
}

int bwd_chunk() { return kQ; }
int bwd_max_headdim() { return kPMax; }

cudaError_t launch_bwd(const BwdProblem& q, void* workspace, cudaStream_t s) {
  const BwdWs w = bwd_ws(q.fwd);
  char* ws = static_cast<char*>(workspace);
  return q.fwd.io == SSD_DTYPE_BF16 ? run_bwd_t<__nv_bfloat16>(q, w, ws, s) : run_bwd_t<float>(q, w, ws, s);
}

}  // namespace ssd
