// bwd.cu -- gradient of the SSD forward pass: the driver of both paths, the
// two state recurrences, and the fp32 CUDA-core gradient kernel (io fp32 or
// bf16, chunk 64; the bf16 headdim-64 dstate-128 path uses bwd_tc.cu).
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
#include <cstdlib>
#include <type_traits>

#include "internal.h"

namespace ssd {
namespace {

constexpr int kQ = 64;    // chunk length of the CUDA-core gradient kernel
constexpr int kT = 256;   // threads per block
constexpr int kNT = 32;   // state columns per slice
constexpr int kPMax = 128;
constexpr int kQTc = 128;  // chunk length of the tensor-core gradient kernel

__device__ __forceinline__ float ld_f(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_f(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_f(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_f(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

template <typename V>
__device__ __forceinline__ V vzero();
template <>
__device__ __forceinline__ float vzero<float>() { return 0.f; }
template <>
__device__ __forceinline__ float4 vzero<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }
__device__ __forceinline__ float vfma(float a, float x, float y) { return fmaf(a, x, y); }
__device__ __forceinline__ float4 vfma(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}
__device__ __forceinline__ void store_bf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
__device__ __forceinline__ void store_bf(__nv_bfloat16* p, float4 v) {  // 8-byte aligned
  __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// ---------------------------------------------------------------------------
// The adjoint recurrence across chunks, last chunk first.  On entry slot c
// holds dS_c; on exit it holds Gout[c] (or, with gout_bf, Gout[c] goes to
// gout_bf as bf16 and slot c is left as it was), and dinit = the G entering
// chunk 0.
// One thread per state entry.
// ---------------------------------------------------------------------------
template <int VEC>
__global__ void __launch_bounds__(kT) bwd_state_passing_kernel(const float* __restrict__ dA_cs,
                                                               const float* __restrict__ dfinal,
                                                               float* __restrict__ gstates,
                                                               float* __restrict__ dinit, int64_t H,
                                                               int64_t PN, int64_t nc, int Q,
                                                               __nv_bfloat16* __restrict__ gout_bf) {
  using V = typename std::conditional<VEC == 4, float4, float>::type;
  const int64_t e = ((int64_t)blockIdx.x * kT + threadIdx.x) * VEC;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  if (e >= PN) return;
  auto at = [&](float* base, int64_t row) { return reinterpret_cast<V*>(base + row * PN + e); };
  V gv = dfinal ? *reinterpret_cast<const V*>(dfinal + (b * H + h) * PN + e) : vzero<V>();
  const float* cs = dA_cs + (b * H + h) * nc * Q;
  // four chunks per group, loads first; four state entries per thread when
  // VEC = 4 (measured: 2, 4, 8, 16 chunks per group -> the backward pass on
  // the 2.7B-shaped layer 2.115 / 2.108 / 2.161 / 2.487 ms)
  constexpr int U = 4;
  for (int64_t c0 = nc - 1; c0 >= 0; c0 -= U) {
    V ds[U];
    float dec[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 - u;
      ds[u] = c >= 0 ? *at(gstates, (b * nc + c) * H + h) : vzero<V>();
      dec[u] = c >= 0 ? expf(cs[c * Q + Q - 1]) : 1.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 - u;
      if (c >= 0) {
        if (gout_bf)
          store_bf(gout_bf + ((b * nc + c) * H + h) * PN + e, gv);
        else
          *at(gstates, (b * nc + c) * H + h) = gv;
        gv = vfma(dec[u], gv, ds[u]);
      }
    }
  }
  if (dinit) *at(dinit, b * H + h) = gv;
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

// Thread layout of every product below: warp w owns the eight token rows
// r_u = 8w + u of the chunk; lane l owns columns l, l + 32, ... of the
// result.  Row operands are read as 16-byte vectors (the same address for
// the whole warp), column operands one element per lane, so each shared-
// memory load feeds several FMAs.
constexpr int kLdQ = kQ + 4;    // row stride of the Q×Q matrices (16-byte rows)
constexpr int kLdS = kNT + 4;   // row stride of the state slices

template <int PMAX>
struct ChunkSmem {
  static constexpr int kLdP = PMAX + 4;
  static constexpr int kXs = 0;                         // x  [Q][P]
  static constexpr int kDys = kXs + kQ * kLdP;          // dy [Q][P]
  static constexpr int kM2 = kDys + kQ * kLdP;         // e^{cs_s-cs_j} DX[s][j]           (j ≤ s)
  static constexpr int kM3 = kM2 + kQ * kLdQ;           // transposed: [j][s] e^{cs_s-cs_j} Δ_j DX[s][j]
  static constexpr int kBs = kM3 + kQ * kLdQ;           // B slice [Q][NT]
  static constexpr int kCs = kBs + kQ * kLdS;           // C slice [Q][NT]
  static constexpr int kGs = kCs + kQ * kLdS;           // Gout slice [P][NT]
  static constexpr int kHs = kGs + PMAX * kLdS;         // h_in slice [P][NT]
  // e^{cs_s-cs_j} CB[s][j] (j ≤ s): needed only between the two passes over
  // the state slices, so it lives in the slice buffers (two blocks per SM at
  // headdim 64)
  static constexpr int kM1 = kBs;
  static_assert(kQ * kLdQ <= 2 * kQ * kLdS + 2 * PMAX * kLdS, "M1 fits in the slice buffers");
  static constexpr int kVec = kHs + PMAX * kLdS;
  // vectors: cs, dl, xu, gbx, a1, rows, cols, rp (Q+1), red (kT)
  static constexpr int kFloats = kVec + 8 * kQ + 1 + kT;
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T, int PMAX>
__global__ void __launch_bounds__(kT, PMAX <= 64 ? 2 : 1) bwd_chunk_kernel(const ChunkGradArgs a) {
  using S = ChunkSmem<PMAX>;
  constexpr int LDP = S::kLdP;
  constexpr int NPJ = PMAX / 32;  // head-dim columns per lane
  extern __shared__ __align__(16) float sm[];
  float* xs = sm + S::kXs;
  float* dys = sm + S::kDys;
  float* M1 = sm + S::kM1;
  float* M2 = sm + S::kM2;
  float* M3T = sm + S::kM3;
  float* Bs = sm + S::kBs;
  float* Cs = sm + S::kCs;
  float* Gs = sm + S::kGs;
  float* Hs = sm + S::kHs;
  float* cs = sm + S::kVec;
  float* dl = cs + kQ;
  float* xu = dl + kQ;      // x_t·u_t
  float* gbx = xu + kQ;     // x_t·(Gout B_t)
  float* a1 = gbx + kQ;     // e^{cs_t} C_t·(h_inᵀ dy_t)
  float* rows = a1 + kQ;    // Σ_{j<k} W[k][j]
  float* cols = rows + kQ;  // Σ_{s>k} W[s][k]
  float* rp = cols + kQ;    // [Q+1]
  float* red = rp + kQ + 1; // [kT]

  const T* x = static_cast<const T*>(a.x);
  const T* dy = static_cast<const T*>(a.dy);
  const T* Bm = static_cast<const T*>(a.Bm);
  const T* Cm = static_cast<const T*>(a.Cm);
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (a.H / a.G);
  const int P = a.P, N = a.N;
  const int P4 = (P + 3) & ~3;
  const int tid = threadIdx.x, lane = tid & 31, w8 = (tid >> 5) * 8;
  const int64_t t0 = c * kQ;

  for (int i = tid; i < kQ; i += kT) {
    cs[i] = a.dA_cs[((b * a.H + h) * a.nc + c) * kQ + i];
    dl[i] = a.dt_c[((b * a.H + h) * a.nc + c) * kQ + i];
    a1[i] = 0.f;
    cols[i] = 0.f;
  }
  // all PMAX columns: the lanes whose columns lie past P read zeros
  for (int e = tid; e < kQ * PMAX; e += kT) {
    const int i = e / PMAX, p = e - i * PMAX;
    const int64_t t = t0 + i;
    const bool ok = t < a.L && p < P;
    const int64_t o = ((b * a.L + t) * a.H + h) * P + p;
    xs[i * LDP + p] = ok ? ld_f(x, o) : 0.f;
    dys[i * LDP + p] = ok ? ld_f(dy, o) : 0.f;
  }
  __syncthreads();
  // DX[s][j] = dy_s·x_j for s = r_u, j = lane, lane + 32
  float dxr[8][2];
#pragma unroll
  for (int u = 0; u < 8; ++u) dxr[u][0] = dxr[u][1] = 0.f;
  for (int p = 0; p < P4; p += 4) {
    const float4 x0 = *reinterpret_cast<const float4*>(xs + lane * LDP + p);
    const float4 x1 = *reinterpret_cast<const float4*>(xs + (lane + 32) * LDP + p);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 yv = *reinterpret_cast<const float4*>(dys + (w8 + u) * LDP + p);
      dxr[u][0] += dot4(yv, x0);
      dxr[u][1] += dot4(yv, x1);
    }
  }
  // CB[s][j] = C_s·B_j and GB[t][p] = Σ_n B_t[n] Gout[p][n] over state
  // slices; γ = <Gout, h_in>
  float cb[8][2], gb[8][NPJ];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    cb[u][0] = cb[u][1] = 0.f;
#pragma unroll
    for (int v = 0; v < NPJ; ++v) gb[u][v] = 0.f;
  }
  float gam = 0.f;
  const float* hin = a.states + ((b * a.nc + c) * a.H + h) * (int64_t)P * N;
  const float* gout = a.gstates + ((b * a.nc + c) * a.H + h) * (int64_t)P * N;
  auto load_slices = [&](int n0) {
    for (int e = tid; e < kQ * kNT; e += kT) {
      const int i = e / kNT, k = e - i * kNT;
      const int64_t t = t0 + i;
      const bool ok = t < a.L && n0 + k < N;
      const int64_t o = ((b * a.L + t) * a.G + g) * N + n0 + k;
      Bs[i * kLdS + k] = ok ? ld_f(Bm, o) : 0.f;
      Cs[i * kLdS + k] = ok ? ld_f(Cm, o) : 0.f;
    }
    for (int e = tid; e < PMAX * kNT; e += kT) {
      const int p = e / kNT, k = e - p * kNT;
      const bool ok = p < P && n0 + k < N;
      Gs[p * kLdS + k] = ok ? gout[(int64_t)p * N + n0 + k] : 0.f;
      Hs[p * kLdS + k] = ok ? hin[(int64_t)p * N + n0 + k] : 0.f;
    }
  };
  for (int n0 = 0; n0 < N; n0 += kNT) {
    __syncthreads();
    load_slices(n0);
    __syncthreads();
#pragma unroll 2
    for (int k = 0; k < kNT; k += 4) {
      const float4 b0 = *reinterpret_cast<const float4*>(Bs + lane * kLdS + k);
      const float4 b1 = *reinterpret_cast<const float4*>(Bs + (lane + 32) * kLdS + k);
      float4 gp[NPJ];
#pragma unroll
      for (int v = 0; v < NPJ; ++v) gp[v] = *reinterpret_cast<const float4*>(Gs + (lane + 32 * v) * kLdS + k);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 cv = *reinterpret_cast<const float4*>(Cs + (w8 + u) * kLdS + k);
        const float4 bv = *reinterpret_cast<const float4*>(Bs + (w8 + u) * kLdS + k);
        cb[u][0] += dot4(cv, b0);
        cb[u][1] += dot4(cv, b1);
#pragma unroll
        for (int v = 0; v < NPJ; ++v) gb[u][v] += dot4(bv, gp[v]);
      }
    }
    for (int e = tid; e < P * kNT; e += kT) {
      const int p = e / kNT, k = e - p * kNT;
      gam = fmaf(Gs[p * kLdS + k], Hs[p * kLdS + k], gam);
    }
  }
  // Masked matrices, the strict row/column sums of W = M3 ⊙ CB, and dD (the
  // trace of DX).  M1 overwrites the slice buffers: every warp is done with them.
  __syncthreads();
  float ddsum = 0.f, colacc[2] = {0.f, 0.f};
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int s = w8 + u;
    float rowacc = 0.f;
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int j = lane + 32 * jj;
      const float dxv = dxr[u][jj];
      if (s == j) ddsum += dxv;
      const float E = j <= s ? expf(cs[s] - cs[j]) : 0.f;
      const float wc = E * dl[j] * dxv;
      M1[s * kLdQ + j] = E * cb[u][jj];
      M2[s * kLdQ + j] = E * dxv;
      M3T[j * kLdQ + s] = wc;
      if (j < s) {
        const float W = wc * cb[u][jj];
        rowacc += W;
        colacc[jj] += W;
      }
    }
    rowacc = warp_sum(rowacc);
    if (lane == 0) rows[s] = rowacc;
  }
  atomicAdd(&cols[lane], colacc[0]);
  atomicAdd(&cols[lane + 32], colacc[1]);
  __syncthreads();
  const float cs_last = cs[kQ - 1];
  // u_t = Σ_{s≥t} M1[s][t] dy_s + e^{cs_last-cs_t} GB[t];  dx_t = D dy_t + Δ_t u_t
  {
    float ua[8][NPJ];
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < NPJ; ++v) ua[u][v] = 0.f;
    for (int s = w8; s < kQ; ++s) {
      const float4 m0 = *reinterpret_cast<const float4*>(M1 + s * kLdQ + w8);
      const float4 m1 = *reinterpret_cast<const float4*>(M1 + s * kLdQ + w8 + 4);
      const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int v = 0; v < NPJ; ++v) {
        const float dv = dys[s * LDP + lane + 32 * v];
#pragma unroll
        for (int u = 0; u < 8; ++u) ua[u][v] = fmaf(mu[u], dv, ua[u][v]);
      }
    }
    const float Dh = a.D ? a.D[h] : 0.f;
    T* dxo = static_cast<T*>(a.dx);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = w8 + u;
      const float eg = expf(cs_last - cs[t]);
      const int64_t tt = t0 + t;
      float xuv = 0.f, gbv = 0.f;
#pragma unroll
      for (int v = 0; v < NPJ; ++v) {
        const int p = lane + 32 * v;
        const float uu = fmaf(eg, gb[u][v], ua[u][v]);
        const float xv = xs[t * LDP + p];
        xuv = fmaf(xv, uu, xuv);
        gbv = fmaf(xv, gb[u][v], gbv);
        if (tt < a.L && p < P) st_f(dxo, ((b * a.L + tt) * a.H + h) * P + p, fmaf(Dh, dys[t * LDP + p], dl[t] * uu));
      }
      xuv = warp_sum(xuv);
      gbv = warp_sum(gbv);
      if (lane == 0) {
        xu[t] = xuv;
        gbx[t] = gbv;
      }
    }
  }
  // dB and dC over state slices; a1_t = e^{cs_t} C_t·(h_inᵀ dy_t)
  for (int n0 = 0; n0 < N; n0 += kNT) {
    __syncthreads();
    load_slices(n0);
    __syncthreads();
    float xg[8], yh[8], vb[8], vc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) xg[u] = yh[u] = vb[u] = vc[u] = 0.f;
    for (int p = 0; p < P4; p += 4) {
      const float g0 = Gs[p * kLdS + lane], g1 = Gs[(p + 1) * kLdS + lane];
      const float g2 = Gs[(p + 2) * kLdS + lane], g3 = Gs[(p + 3) * kLdS + lane];
      const float h0 = Hs[p * kLdS + lane], h1 = Hs[(p + 1) * kLdS + lane];
      const float h2 = Hs[(p + 2) * kLdS + lane], h3 = Hs[(p + 3) * kLdS + lane];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float4 xv = *reinterpret_cast<const float4*>(xs + (w8 + u) * LDP + p);
        const float4 yv = *reinterpret_cast<const float4*>(dys + (w8 + u) * LDP + p);
        xg[u] = fmaf(xv.x, g0, fmaf(xv.y, g1, fmaf(xv.z, g2, fmaf(xv.w, g3, xg[u]))));
        yh[u] = fmaf(yv.x, h0, fmaf(yv.y, h1, fmaf(yv.z, h2, fmaf(yv.w, h3, yh[u]))));
      }
    }
    for (int s = w8; s < kQ; ++s) {
      const float cv = Cs[s * kLdS + lane];
      const float4 m0 = *reinterpret_cast<const float4*>(M2 + s * kLdQ + w8);
      const float4 m1 = *reinterpret_cast<const float4*>(M2 + s * kLdQ + w8 + 4);
      vb[0] = fmaf(m0.x, cv, vb[0]);
      vb[1] = fmaf(m0.y, cv, vb[1]);
      vb[2] = fmaf(m0.z, cv, vb[2]);
      vb[3] = fmaf(m0.w, cv, vb[3]);
      vb[4] = fmaf(m1.x, cv, vb[4]);
      vb[5] = fmaf(m1.y, cv, vb[5]);
      vb[6] = fmaf(m1.z, cv, vb[6]);
      vb[7] = fmaf(m1.w, cv, vb[7]);
    }
    for (int j = 0; j < w8 + 8; ++j) {
      const float bv = Bs[j * kLdS + lane];
      const float4 m0 = *reinterpret_cast<const float4*>(M3T + j * kLdQ + w8);
      const float4 m1 = *reinterpret_cast<const float4*>(M3T + j * kLdQ + w8 + 4);
      vc[0] = fmaf(m0.x, bv, vc[0]);
      vc[1] = fmaf(m0.y, bv, vc[1]);
      vc[2] = fmaf(m0.z, bv, vc[2]);
      vc[3] = fmaf(m0.w, bv, vc[3]);
      vc[4] = fmaf(m1.x, bv, vc[4]);
      vc[5] = fmaf(m1.y, bv, vc[5]);
      vc[6] = fmaf(m1.z, bv, vc[6]);
      vc[7] = fmaf(m1.w, bv, vc[7]);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int t = w8 + u;
      const float ecs = expf(cs[t]);
      const float db = dl[t] * fmaf(expf(cs_last - cs[t]), xg[u], vb[u]);
      const float dc = fmaf(ecs, yh[u], vc[u]);
      const float a1v = warp_sum(ecs * Cs[t * kLdS + lane] * yh[u]);
      if (lane == 0) a1[t] += a1v;
      const int64_t tt = t0 + t;
      if (tt < a.L && n0 + lane < N) {
        const int64_t o = ((b * a.L + tt) * a.G + g) * N + n0 + lane;
        atomicAdd(a.dB_acc + o, db);
        atomicAdd(a.dC_acc + o, dc);
      }
    }
  }
  // rp[t] = Σ_{s≥t} Σ_{j<t} W[s][j], from rp[k+1] - rp[k] = cols[k] - rows[k]
  for (int k = tid; k < kQ; k += kT) rp[k + 1] = cols[k] - rows[k];
  if (tid == 0) rp[0] = 0.f;
  red[tid] = gam;
  __syncthreads();
  if (tid < 32) {
    float v = 0.f;
    for (int i = tid; i < kT; i += 32) v += red[i];
    v = warp_sum(v);
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
    v = warp_sum(v);
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
cudaError_t run_bwd_t(const BwdProblem& qin, const BwdWs& w, char* ws, cudaStream_t s) {
  BwdProblem q = qin;
  q.fwd.err = reinterpret_cast<int32_t*>(ws);  // status word, cleared below
  const Problem& p = q.fwd;
  float* dA_cs = reinterpret_cast<float*>(ws + w.off_cs);
  float* dt_c = reinterpret_cast<float*>(ws + w.off_dt);
  float* states = reinterpret_cast<float*>(ws + w.off_states);
  float* gstates = reinterpret_cast<float*>(ws + w.off_gstates);
  float* dB_acc = reinterpret_cast<float*>(ws + w.off_db);
  float* dC_acc = reinterpret_cast<float*>(ws + w.off_dc);
  const int64_t nbc = p.B * p.L * p.G * p.N;
  cudaError_t e;
  if ((e = cudaMemsetAsync(p.err, 0, sizeof(int32_t), s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dB_acc, 0, (size_t)nbc * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(dC_acc, 0, (size_t)nbc * 4, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(q.dA, 0, (size_t)p.H * 4, s)) != cudaSuccess) return e;
  if (q.dD && (e = cudaMemsetAsync(q.dD, 0, (size_t)p.H * 4, s)) != cudaSuccess) return e;
  // Tensor-core path: the states entering (h_in) and the adjoints leaving
  // (Gout) each chunk go to bf16 copies in the two halves of the gstates
  // region, and the fp32 region `states` is reused for the adjoint chunk
  // states.  Otherwise h_in stays fp32 in `states`, Gout fp32 in `gstates`.
  const bool tc = p.Q == kQTc;
  const int64_t nst = p.B * p.nc * p.H * p.P * p.N;
  __nv_bfloat16* hin_bf = tc ? reinterpret_cast<__nv_bfloat16*>(gstates) : nullptr;
  __nv_bfloat16* gout_bf = tc ? hin_bf + nst : nullptr;
  float* adj = tc ? states : gstates;
  if ((e = launch_chunk_cumsum(p, dA_cs, dt_c, s)) != cudaSuccess) return e;
  if (bwd_walks(p)) {
    // tensor-core path: the forward states and the adjoint states, each a
    // walk of the fused path's states kernel over whole sequences (the
    // adjoint last chunk first), the state on chip and only its bf16 copies
    // (and dinit) written; both kinds of walk in one launch
    uint32_t* wflag = reinterpret_cast<uint32_t*>(ws + w.off_wflag);
    if ((e = cudaMemsetAsync(wflag, 0, w.off_wslot - w.off_wflag, s)) != cudaSuccess) return e;
    if ((e = launch_states_walks(p, hin_bf, q.dy, q.dfinal, q.dinit, gout_bf, wflag,
                                 reinterpret_cast<float*>(ws + w.off_wslot), p.err, s)) != cudaSuccess)
      return e;
  } else {
    // forward recompute: chunk states, then the recurrence (the state
    // entering each chunk)
    if ((e = launch_chunk_state(p, dA_cs, dt_c, states, s)) != cudaSuccess) return e;
    if ((e = launch_state_passing(p, dA_cs, states, s, hin_bf)) != cudaSuccess) return e;
    // adjoint chunk states, then the adjoint recurrence (last chunk first)
    if ((e = launch_chunk_state_adjoint(p, q.dy, dA_cs, adj, s)) != cudaSuccess) return e;
    const int64_t PN = p.P * p.N;
    dim3 grid((unsigned)((PN + kT - 1) / kT), (unsigned)p.H, (unsigned)p.B);
    if (PN % 4 == 0) {
      dim3 g4((unsigned)((PN / 4 + kT - 1) / kT), (unsigned)p.H, (unsigned)p.B);
      bwd_state_passing_kernel<4><<<g4, kT, 0, s>>>(dA_cs, q.dfinal, adj, q.dinit, p.H, PN, p.nc, (int)p.Q, gout_bf);
    } else {
      bwd_state_passing_kernel<1><<<grid, kT, 0, s>>>(dA_cs, q.dfinal, adj, q.dinit, p.H, PN, p.nc, (int)p.Q,
                                                      gout_bf);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const unsigned cgrid = (unsigned)std::min<int64_t>((nbc + kT - 1) / kT, 4096);
  if (tc) {
    if ((e = launch_bwd_chunk_tc(q, dA_cs, dt_c, hin_bf, gout_bf, dB_acc, dC_acc, s)) != cudaSuccess) return e;
    bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dB_acc, (T*)q.dBm, nbc);
    bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dC_acc, (T*)q.dCm, nbc);
    return cudaGetLastError();
  }
  if (p.Q != kQ) return cudaErrorInvalidValue;
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
  bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dB_acc, (T*)q.dBm, nbc);
  bwd_convert_kernel<T><<<cgrid, kT, 0, s>>>(dC_acc, (T*)q.dCm, nbc);
  return cudaGetLastError();
}

}  // namespace

// Both state recurrences of the backward pass as walks of the fused path's
// states kernel: the tensor-core path (chunk 128: bf16, headdim 64, dstate
// 128) within the kernel's index range.
bool bwd_walks(const Problem& p) {
  return p.Q == kQTc && p.B * p.H < (int64_t(1) << 24) && p.L < (int64_t(1) << 30);
}

BwdWs bwd_ws(const Problem& p) {
  BwdWs w;
  const size_t ncs = align_up((size_t)(p.B * p.H * p.nc * p.Q) * 4, 256);
  const size_t nst = align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 4, 256);
  const size_t nbc = align_up((size_t)(p.B * p.L * p.G * p.N) * 4, 256);
  // the fp32 per-chunk states are not needed where both state recurrences
  // are walks of the states kernel (tensor-core path), which write only the
  // bf16 copies (h_in and Gout, in the gstates region)
  const bool walks = bwd_walks(p);
  w.off_cs = 256;  // the first 256 bytes hold the status word
  w.off_dt = w.off_cs + ncs;
  w.off_states = w.off_dt + ncs;
  w.off_gstates = w.off_states + (walks ? 0 : nst);
  w.off_db = w.off_gstates + nst;
  w.off_dc = w.off_db + nbc;
  // the state walks' hand-offs: a flag and an fp32 state per walk and head
  const size_t nw = walks ? (size_t)states_walks(p) * 2 : 0;
  w.off_wflag = w.off_dc + nbc;
  w.off_wslot = w.off_wflag + align_up(nw * 4, 256);
  w.total = w.off_wslot + align_up(nw * p.P * p.N * 4, 256);
  return w;
}

int bwd_chunk(const Problem& p, int64_t requested) {
  const char* env = getenv("SSD_BWD_CUDA_CORES");
  const bool tc = bwd_tc_supported(p) && !(env && atoi(env) == 1);
  if (requested == 0) return tc ? kQTc : kQ;
  if (requested == kQ) return kQ;
  if (requested == kQTc && tc) return kQTc;
  return 0;
}
int bwd_max_headdim() { return kPMax; }

cudaError_t launch_bwd(const BwdProblem& q, void* workspace, cudaStream_t s) {
  const BwdWs w = bwd_ws(q.fwd);
  char* ws = static_cast<char*>(workspace);
  return q.fwd.io == SSD_DTYPE_BF16 ? run_bwd_t<__nv_bfloat16>(q, w, ws, s) : run_bwd_t<float>(q, w, ws, s);
}

}  // namespace ssd
