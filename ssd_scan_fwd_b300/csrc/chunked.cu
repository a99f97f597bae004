// chunked.cu -- the four step kernels of the chunked SSD forward pass on
// CUDA cores (fp32 arithmetic, fp32 or bf16 io), and the launchers that send
// the chunk states and outputs of bf16 headdim-64 problems to the tensor-core
// kernels of state_tc.cu and scan_tc.cu.
//
// This path serves fp32 problems (tensor-core formats cannot hold fp32
// accuracy), any head/state size up to 256, and the per-step entry points
// whose intermediates the tests compare with the oracle's chunked form.
//
// The decomposition (page "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进",
// §2.1.2 recurrence, §2.2.1 masked matrix form, §2.2.2 block decomposition):
//   chunk_cumsum   cs_i = Σ_{k≤i} Δ_k A_h inside each chunk
//   chunk_state    S_c = Σ_i exp(cs_{Q-1} − cs_i) Δ_i x_i B_iᵀ
//   state_passing  h_in[c+1] = exp(cs_{c,Q-1}) h_in[c] + S_c
//   chunk_scan     y_i = Σ_{j≤i} (C_i·B_j) exp(cs_i − cs_j) Δ_j x_j
//                        + exp(cs_i) C_iᵀ h_in[c] + D x_i
// The mask exp(cs_i − cs_j) is only evaluated for j ≤ i, where the exponent
// is ≤ 0 (A ≤ 0, Δ ≥ 0), so it never overflows.

#include <cuda_bf16.h>

#include <cstdlib>
#include <type_traits>

#include "internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

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
// Step 1: in-chunk inclusive sums of log α = Δ·A.  One block per
// (chunk, block of heads, batch); one thread per token of the chunk.
// ---------------------------------------------------------------------------
// Δ from the raw dt: + dt_bias[h] when given, then softplus when asked
// (softplus(v) = log(1 + e^v); for v > 20 it equals v to fp32 precision).
__device__ __forceinline__ float make_delta(float v, const float* dt_bias, int softplus, int64_t h) {
  if (dt_bias) v += dt_bias[h];
  if (softplus) v = v > 20.f ? v : log1pf(expf(v));
  return v;
}

// With theta (the complex decay's rotation angles, [B][L][H]) the in-chunk
// sums φ_i = Σ_{k≤i} θ_k go to phi in the same layout.
template <int Q>
__global__ void __launch_bounds__(Q) chunk_cumsum_kernel(const float* __restrict__ dt,
                                                         const float* __restrict__ dt_bias, int softplus,
                                                         const float* __restrict__ A,
                                                         const float* __restrict__ theta,
                                                         int64_t L, int64_t H, int64_t nc,
                                                         int heads_per_block,
                                                         float* __restrict__ dA_cs,
                                                         float* __restrict__ dt_c,
                                                         float* __restrict__ phi) {
  __shared__ float warp_total[Q / 32];
  const int64_t c = blockIdx.x;
  const int64_t b = blockIdx.z;
  const int i = threadIdx.x;
  const int lane = i & 31, warp = i >> 5;
  const int64_t t = c * Q + i;
  const int64_t h_begin = (int64_t)blockIdx.y * heads_per_block;
  const int64_t h_end = min(h_begin + heads_per_block, H);
  // inclusive sum over the chunk (threads in token order)
  auto block_scan = [&](float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float up = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += up;
    }
    if (lane == 31) warp_total[warp] = v;
    __syncthreads();
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off += warp_total[w];
    __syncthreads();
    return v + off;
  };
  for (int64_t h = h_begin; h < h_end; ++h) {
    const float d = (t < L) ? make_delta(dt[(b * L + t) * H + h], dt_bias, softplus, h) : 0.f;
    const float v = block_scan(d * A[h]);
    const int64_t o = ((b * H + h) * nc + c) * Q + i;
    dA_cs[o] = v;
    dt_c[o] = d;
    if (theta) phi[o] = block_scan(t < L ? theta[(b * L + t) * H + h] : 0.f);
  }
}

// ---------------------------------------------------------------------------
// Step 2: chunk states S_c[p][n] = Σ_i w_i x_i[p] B_i[n],
// w_i = exp(cs_{Q-1} − cs_i) Δ_i.  One block per (chunk, head, batch).
// The weight w_i by mode: kFwd the above; kAdjoint exp(cs_i) (the backward
// pass's adjoint chunk states Σ_i exp(cs_i) dy_i[p] C_i[n], x := dy,
// B := C); kRotRe / kRotIm exp(cs_{Q-1} − cs_i) cos / sin(φ_{Q-1} − φ_i) Δ_i,
// the real and imaginary chunk states of the complex decay (φ the in-chunk
// sums of the rotation angles).
// Warp w owns state rows p0 + 8w .. p0 + 8w + 7 of a 64 × 128 output tile,
// lane l the columns n0 + l + 32v: each token's row operand comes as two
// 16-byte loads shared by the warp, its four column operands one per lane.
// Registers are capped for four blocks per SM (the loads of one block overlap
// the arithmetic of the others; measured 2.0 -> 1.6 ms per launch on the
// 2.7B-shaped layer).
// ---------------------------------------------------------------------------
enum : int { kFwd = 0, kAdjoint = 1, kRotRe = 2, kRotIm = 3 };

template <typename T, int Q, int kMode>
__global__ void __launch_bounds__(kThreads, 4) chunk_state_kernel(
    const T* __restrict__ x, const T* __restrict__ Bm, const float* __restrict__ dA_cs,
    const float* __restrict__ dt_c, const float* __restrict__ phi, int64_t L, int64_t H, int P, int G, int N,
    int64_t nc, float* __restrict__ states) {
  constexpr int PT = 64, NT = 128;
  constexpr int LA = PT + 4, LB = NT + 4;
  extern __shared__ __align__(16) float smem[];
  float* as = smem;           // [Q][PT+4]: rows x_i scaled by w_i
  float* bs = smem + Q * LA;  // [Q][NT+4]
  __shared__ float w_s[Q];
  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t g = h / (H / G);
  const int tid = threadIdx.x, lane = tid & 31, w8 = (tid >> 5) * 8;
  const float* cs = dA_cs + ((b * H + h) * nc + c) * Q;
  const float* dl = kMode == kAdjoint ? nullptr : dt_c + ((b * H + h) * nc + c) * Q;
  const float* ph = (kMode == kRotRe || kMode == kRotIm) ? phi + ((b * H + h) * nc + c) * Q : nullptr;
  for (int i = tid; i < Q; i += kThreads) {
    if (kMode == kAdjoint) {
      w_s[i] = expf(cs[i]);
    } else if (kMode == kFwd) {
      w_s[i] = expf(cs[Q - 1] - cs[i]) * dl[i];
    } else {
      const float a = ph[Q - 1] - ph[i];
      w_s[i] = expf(cs[Q - 1] - cs[i]) * dl[i] * (kMode == kRotRe ? cosf(a) : sinf(a));
    }
  }
  float* out = states + ((b * nc + c) * H + h) * (int64_t)P * N;
  for (int p0 = 0; p0 < P; p0 += PT) {
    for (int n0 = 0; n0 < N; n0 += NT) {
      __syncthreads();
      for (int e = tid; e < Q * PT; e += kThreads) {
        const int i = e / PT, p = e - i * PT;
        const int64_t t = c * Q + i;
        as[i * LA + p] = (t < L && p0 + p < P) ? to_f(x[((b * L + t) * H + h) * P + p0 + p]) * w_s[i] : 0.f;
      }
      for (int e = tid; e < Q * NT; e += kThreads) {
        const int i = e / NT, n = e - i * NT;
        const int64_t t = c * Q + i;
        bs[i * LB + n] = (t < L && n0 + n < N) ? to_f(Bm[((b * L + t) * G + g) * N + n0 + n]) : 0.f;
      }
      __syncthreads();
      float acc[8][4];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
#pragma unroll 4
      for (int i = 0; i < Q; ++i) {
        const float4 a0 = *reinterpret_cast<const float4*>(as + i * LA + w8);
        const float4 a1 = *reinterpret_cast<const float4*>(as + i * LA + w8 + 4);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float bv[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) bv[v] = bs[i * LB + lane + 32 * v];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + w8 + u;
        if (p >= P) continue;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int n = n0 + lane + 32 * v;
          if (n < N) out[(int64_t)p * N + n] = acc[u][v];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Step 3: the state recurrence across chunks.  One thread per state entry;
// sequential over chunks.  states[c] := state entering chunk c.
// ---------------------------------------------------------------------------
// VEC = 4: four consecutive state entries per thread with 16-byte accesses
// (P·N a multiple of 4); VEC = 1 otherwise.
template <int VEC>
__global__ void __launch_bounds__(kThreads) state_passing_kernel(
    const float* __restrict__ dA_cs, const float* init, float* __restrict__ states,
    float* final_state, int64_t H, int64_t PN, int64_t nc, int Q, __nv_bfloat16* __restrict__ states_bf) {
  using V = typename std::conditional<VEC == 4, float4, float>::type;
  const int64_t e = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * VEC;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  if (e >= PN) return;
  auto at = [&](float* base, int64_t row) { return reinterpret_cast<V*>(base + row * PN + e); };
  // the state entering chunk c: fp32 in place, or (states_bf) bf16 to its own buffer
  auto put = [&](int64_t row, const V& v) {
    if (states_bf)
      store_bf(states_bf + row * PN + e, v);
    else
      *at(states, row) = v;
  };
  V s = init ? *reinterpret_cast<const V*>(init + (b * H + h) * PN + e) : vzero<V>();
  const float* cs = dA_cs + (b * H + h) * nc * Q;
  // eight chunks per group: their loads are all in flight before the
  // dependent updates run
  constexpr int U = 8;
  for (int64_t c0 = 0; c0 < nc; c0 += U) {
    V sc[U];
    float dec[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u;
      sc[u] = c < nc ? *at(states, (b * nc + c) * H + h) : vzero<V>();
      dec[u] = c < nc ? expf(cs[c * Q + Q - 1]) : 1.f;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u;
      if (c < nc) {
        put((b * nc + c) * H + h, s);
        s = vfma(dec[u], s, sc[u]);
      }
    }
  }
  if (final_state) *at(final_state, b * H + h) = s;
}

// ---------------------------------------------------------------------------
// Step 4: outputs of each chunk.  One block per (chunk, head × p-tile, batch).
// kRot (complex decay): the mask gains cos(φ_i − φ_j) and the read-out is
// Re(e^{iφ_i} h_in) = cos φ_i Re h_in − sin φ_i Im h_in.
// Every product is register-tiled: warp w owns the Q/8 token rows
// i = w·Q/8 .. of the chunk, lane l the columns l + 32v of the result; the
// row operand of a step is a 16-byte shared-memory load common to the warp.
// Up to chunk 64, registers are capped for three blocks per SM (measured
// 7.4 -> 6.7 ms for the whole chunked pass on the 2.7B-shaped layer).
// ---------------------------------------------------------------------------
template <int Q, bool kRot>
struct ScanSmem {
  static constexpr int PT = 64, NT = 32;
  static constexpr int LQ = Q + 4, LP = PT + 4, LS = NT + 4;
  static constexpr int kMt = 0;                    // [j][i]: masked C Bᵀ, transposed
  static constexpr int kXs = kMt + Q * LQ;         // [Q][PT]
  static constexpr int kCs = kXs + Q * LP;         // C slice [Q][NT]
  static constexpr int kBs = kCs + Q * LS;         // B slice [Q][NT]
  static constexpr int kHs = kBs + Q * LS;         // state slice [PT][NT]
  static constexpr int kHi = kHs + PT * LS;        // imaginary state slice (kRot)
  static constexpr int kVec = kHi + (kRot ? PT * LS : 0);
  static constexpr int kFloats = kVec + 3 * Q;     // cs, Δ, φ
  static constexpr size_t kBytes = sizeof(float) * (size_t)kFloats;
};

template <typename T, int Q, bool kRot>
__global__ void __launch_bounds__(kThreads, Q <= 64 ? 3 : 1) chunk_scan_kernel(
    const T* __restrict__ x, const T* __restrict__ Bm, const T* __restrict__ Cm,
    const float* __restrict__ D, const float* __restrict__ dA_cs, const float* __restrict__ dt_c,
    const float* __restrict__ states, const float* __restrict__ phi, const float* __restrict__ states_im,
    int64_t L, int64_t H, int P, int G, int N, int64_t nc, const T* __restrict__ z, T* __restrict__ y) {
  using S = ScanSmem<Q, kRot>;
  constexpr int PT = S::PT, NT = S::NT, LQ = S::LQ, LP = S::LP, LS = S::LS;
  constexpr int RW = Q / 8;    // token rows per warp
  constexpr int CQ = Q / 32;   // key columns per lane
  constexpr int CP = PT / 32;  // head-dim columns per lane
  extern __shared__ __align__(16) float sm[];
  float* Mt = sm + S::kMt;
  float* xs = sm + S::kXs;
  float* cs_s = sm + S::kCs;
  float* bs_s = sm + S::kBs;
  float* hs = sm + S::kHs;
  float* hsi = sm + S::kHi;
  float* csum = sm + S::kVec;
  float* dls = csum + Q;
  float* phs = dls + Q;

  const int64_t c = blockIdx.x, b = blockIdx.z;
  const int64_t h = blockIdx.y % H;
  const int p0 = (int)(blockIdx.y / H) * PT;
  const int64_t g = h / (H / G);
  const int tid = threadIdx.x, lane = tid & 31, r0 = (tid >> 5) * RW;
  const int64_t t0 = c * Q;

  for (int i = tid; i < Q; i += kThreads) {
    csum[i] = dA_cs[((b * H + h) * nc + c) * Q + i];
    dls[i] = dt_c[((b * H + h) * nc + c) * Q + i];
    phs[i] = kRot ? phi[((b * H + h) * nc + c) * Q + i] : 0.f;
  }
  auto load_cb = [&](int n0, bool with_b) {
    for (int e = tid; e < Q * NT; e += kThreads) {
      const int i = e / NT, k = e - i * NT;
      const int64_t t = t0 + i;
      const bool ok = (t < L) && (n0 + k < N);
      const int64_t off = ((b * L + t) * G + g) * N + n0 + k;
      cs_s[i * LS + k] = ok ? to_f(Cm[off]) : 0.f;
      if (with_b) bs_s[i * LS + k] = ok ? to_f(Bm[off]) : 0.f;
    }
  };
  // S = C Bᵀ over state slices: rows r0 + u, key columns lane + 32v
  float sacc[RW][CQ];
#pragma unroll
  for (int u = 0; u < RW; ++u)
#pragma unroll
    for (int v = 0; v < CQ; ++v) sacc[u][v] = 0.f;
  for (int n0 = 0; n0 < N; n0 += NT) {
    __syncthreads();
    load_cb(n0, true);
    __syncthreads();
#pragma unroll 2
    for (int k = 0; k < NT; k += 4) {
      float4 bv[CQ];
#pragma unroll
      for (int v = 0; v < CQ; ++v) bv[v] = *reinterpret_cast<const float4*>(bs_s + (lane + 32 * v) * LS + k);
#pragma unroll
      for (int u = 0; u < RW; ++u) {
        const float4 cv = *reinterpret_cast<const float4*>(cs_s + (r0 + u) * LS + k);
#pragma unroll
        for (int v = 0; v < CQ; ++v)
          sacc[u][v] = fmaf(cv.x, bv[v].x, fmaf(cv.y, bv[v].y, fmaf(cv.z, bv[v].z, fmaf(cv.w, bv[v].w, sacc[u][v]))));
      }
    }
  }
  // mask: exp(cs_i − cs_j) Δ_j (· cos(φ_i − φ_j)) on and below the diagonal,
  // stored transposed for the next product
#pragma unroll
  for (int u = 0; u < RW; ++u) {
    const int i = r0 + u;
#pragma unroll
    for (int v = 0; v < CQ; ++v) {
      const int j = lane + 32 * v;
      float m = 0.f;
      if (j <= i) {
        m = sacc[u][v] * expf(csum[i] - csum[j]) * dls[j];
        if (kRot) m *= cosf(phs[i] - phs[j]);
      }
      Mt[j * LQ + i] = m;
    }
  }
  for (int e = tid; e < Q * PT; e += kThreads) {
    const int j = e / PT, p = e - j * PT;
    const int64_t t = t0 + j;
    xs[j * LP + p] = (t < L && p0 + p < P) ? to_f(x[((b * L + t) * H + h) * P + p0 + p]) : 0.f;
  }
  __syncthreads();
  // intra-chunk term Y[i][p] = Σ_{j≤i} M[i][j] x_j[p]
  float yacc[RW][CP];
#pragma unroll
  for (int u = 0; u < RW; ++u)
#pragma unroll
    for (int v = 0; v < CP; ++v) yacc[u][v] = 0.f;
  for (int j = 0; j < r0 + RW; ++j) {
    float xv[CP];
#pragma unroll
    for (int v = 0; v < CP; ++v) xv[v] = xs[j * LP + lane + 32 * v];
#pragma unroll
    for (int u4 = 0; u4 < RW; u4 += 4) {
      const float4 m = *reinterpret_cast<const float4*>(Mt + j * LQ + r0 + u4);
      const float mm[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int v = 0; v < CP; ++v) yacc[u4 + q][v] = fmaf(mm[q], xv[v], yacc[u4 + q][v]);
    }
  }
  // read-out of the state entering the chunk: R[i][p] = Σ_n C_i[n] h_in[p][n]
  float racc[RW][CP], racci[RW][CP];
#pragma unroll
  for (int u = 0; u < RW; ++u)
#pragma unroll
    for (int v = 0; v < CP; ++v) racc[u][v] = racci[u][v] = 0.f;
  const float* hin = states + ((b * nc + c) * H + h) * (int64_t)P * N;
  const float* hini = kRot ? states_im + ((b * nc + c) * H + h) * (int64_t)P * N : nullptr;
  for (int n0 = 0; n0 < N; n0 += NT) {
    __syncthreads();
    load_cb(n0, false);
    for (int e = tid; e < PT * NT; e += kThreads) {
      const int p = e / NT, k = e - p * NT;
      const bool ok = p0 + p < P && n0 + k < N;
      hs[p * LS + k] = ok ? hin[(int64_t)(p0 + p) * N + n0 + k] : 0.f;
      if (kRot) hsi[p * LS + k] = ok ? hini[(int64_t)(p0 + p) * N + n0 + k] : 0.f;
    }
    __syncthreads();
#pragma unroll 2
    for (int k = 0; k < NT; k += 4) {
      float4 hv[CP], hvi[CP];
#pragma unroll
      for (int v = 0; v < CP; ++v) {
        hv[v] = *reinterpret_cast<const float4*>(hs + (lane + 32 * v) * LS + k);
        if (kRot) hvi[v] = *reinterpret_cast<const float4*>(hsi + (lane + 32 * v) * LS + k);
      }
#pragma unroll
      for (int u = 0; u < RW; ++u) {
        const float4 cv = *reinterpret_cast<const float4*>(cs_s + (r0 + u) * LS + k);
#pragma unroll
        for (int v = 0; v < CP; ++v) {
          racc[u][v] = fmaf(cv.x, hv[v].x, fmaf(cv.y, hv[v].y, fmaf(cv.z, hv[v].z, fmaf(cv.w, hv[v].w, racc[u][v]))));
          if (kRot)
            racci[u][v] =
                fmaf(cv.x, hvi[v].x, fmaf(cv.y, hvi[v].y, fmaf(cv.z, hvi[v].z, fmaf(cv.w, hvi[v].w, racci[u][v]))));
        }
      }
    }
  }
  const float dh = D ? D[h] : 0.f;
#pragma unroll
  for (int u = 0; u < RW; ++u) {
    const int i = r0 + u;
    const int64_t t = t0 + i;
    const float ecs = expf(csum[i]);
    const float cph = kRot ? cosf(phs[i]) : 1.f, sph = kRot ? sinf(phs[i]) : 0.f;
#pragma unroll
    for (int v = 0; v < CP; ++v) {
      const int p = lane + 32 * v;
      if (t < L && p0 + p < P) {
        const float ro = kRot ? fmaf(cph, racc[u][v], -sph * racci[u][v]) : racc[u][v];
        float val = yacc[u][v] + ecs * ro + dh * xs[i * LP + p];
        const int64_t o = ((b * L + t) * H + h) * P + p0 + p;
        if (z) {  // gate: y · silu(z)
          const float zv = to_f(z[o]);
          val *= zv / (1.f + expf(-zv));
        }
        y[o] = from_f<T>(val);
      }
    }
  }
}

template <int Q, bool kRot>
size_t scan_smem_bytes() {
  return ScanSmem<Q, kRot>::kBytes;
}

template <typename T, int Q, bool kRot>
cudaError_t launch_scan_t(const Problem& p, const float* dA_cs, const float* dt_c,
                          const float* states, const float* phi, const float* states_im, cudaStream_t s) {
  const size_t smem = scan_smem_bytes<Q, kRot>();
  cudaError_t e = cudaFuncSetAttribute(chunk_scan_kernel<T, Q, kRot>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int ptiles = (int)((p.P + 63) / 64);
  dim3 grid((unsigned)p.nc, (unsigned)(p.H * ptiles), (unsigned)p.B);
  chunk_scan_kernel<T, Q, kRot><<<grid, kThreads, smem, s>>>(
      (const T*)p.x, (const T*)p.Bm, (const T*)p.Cm, p.D, dA_cs, dt_c, states, phi, states_im, p.L, p.H,
      (int)p.P, (int)p.G, (int)p.N, p.nc, (const T*)p.z, (T*)p.y);
  return cudaGetLastError();
}

template <typename T, int Q, int kMode>
cudaError_t launch_state_t(const Problem& p, const void* xin, const void* bin, const float* dA_cs,
                           const float* dt_c, const float* phi, float* states, cudaStream_t s) {
  const size_t smem = sizeof(float) * (size_t)Q * ((64 + 4) + (128 + 4));
  cudaError_t e = cudaFuncSetAttribute(chunk_state_kernel<T, Q, kMode>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
  chunk_state_kernel<T, Q, kMode><<<grid, kThreads, smem, s>>>((const T*)xin, (const T*)bin, dA_cs, dt_c, phi,
                                                              p.L, p.H, (int)p.P, (int)p.G, (int)p.N, p.nc,
                                                              states);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Step 3 for the complex decay: h_in[c+1] = e^{cs_last} e^{iφ_last} h_in[c] + S_c
// with S_c = S_re + i S_im; the real and imaginary parts in two arrays.
// ---------------------------------------------------------------------------
template <int VEC>
__global__ void __launch_bounds__(kThreads) state_passing_rot_kernel(
    const float* __restrict__ dA_cs, const float* __restrict__ phi, const float* init_re,
    const float* init_im, float* __restrict__ st_re, float* __restrict__ st_im, float* final_re,
    float* final_im, int64_t H, int64_t PN, int64_t nc, int Q, __nv_bfloat16* __restrict__ re_bf,
    __nv_bfloat16* __restrict__ im_bf) {
  using V = typename std::conditional<VEC == 4, float4, float>::type;
  const int64_t e = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * VEC;
  const int64_t h = blockIdx.y, b = blockIdx.z;
  // Threads past PN stay to the end: the chunk decays are computed by lanes
  // 0..U-1 of each warp and broadcast with shuffles over the whole warp.
  const bool active = e < PN;
  const int lane = threadIdx.x & 31;
  auto at = [&](float* base, int64_t row) { return reinterpret_cast<V*>(base + row * PN + e); };
  V re = active && init_re ? *reinterpret_cast<const V*>(init_re + (b * H + h) * PN + e) : vzero<V>();
  V im = active && init_im ? *reinterpret_cast<const V*>(init_im + (b * H + h) * PN + e) : vzero<V>();
  const float* cs = dA_cs + (b * H + h) * nc * Q;
  const float* ph = phi + (b * H + h) * nc * Q;
  constexpr int U = 8;
  for (int64_t c0 = 0; c0 < nc; c0 += U) {
    V sr[U], si[U];
    float ar[U], ai[U];
    // decay of chunk c0 + lane: e^{cs_last} (cos φ_last + i sin φ_last)
    float my_ar = 1.f, my_ai = 0.f;
    if (lane < U && c0 + lane < nc) {
      const int64_t c = c0 + lane;
      const float mag = expf(cs[c * Q + Q - 1]);
      float sv, cv;
      sincosf(ph[c * Q + Q - 1], &sv, &cv);
      my_ar = mag * cv;
      my_ai = mag * sv;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u;
      const bool ok = active && c < nc;
      sr[u] = ok ? *at(st_re, (b * nc + c) * H + h) : vzero<V>();
      si[u] = ok ? *at(st_im, (b * nc + c) * H + h) : vzero<V>();
      ar[u] = __shfl_sync(0xffffffffu, my_ar, u);
      ai[u] = __shfl_sync(0xffffffffu, my_ai, u);
    }
    if (!active) continue;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t c = c0 + u;
      if (c < nc) {
        const int64_t row = (b * nc + c) * H + h;
        if (re_bf) {  // bf16 copies for the tensor-core chunk outputs
          store_bf(re_bf + row * PN + e, re);
          store_bf(im_bf + row * PN + e, im);
        } else {
          *at(st_re, row) = re;
          *at(st_im, row) = im;
        }
        // (re + i im) · (ar + i ai) + (sr + i si)
        const V nr = vfma(ar[u], re, vfma(-ai[u], im, sr[u]));
        const V ni = vfma(ar[u], im, vfma(ai[u], re, si[u]));
        re = nr;
        im = ni;
      }
    }
  }
  if (!active) return;
  if (final_re) *at(final_re, b * H + h) = re;
  if (final_im) *at(final_im, b * H + h) = im;
}

// bf16 io with headdim 64, dstate 16, 64, 128 or 256, chunk 64 or 128: the
// chunk states on the tensor cores (state_tc.cu).  SSD_CHUNK_STATE_CUDA_CORES=1 keeps them on the
// CUDA-core kernel above (comparisons between the two).
bool use_state_tc(const Problem& p) {
  if (!chunk_state_tc_supported(p)) return false;
  const char* env = getenv("SSD_CHUNK_STATE_CUDA_CORES");
  return !(env && atoi(env) == 1);
}

}  // namespace

cudaError_t launch_rot(const Problem& p, float* dA_cs, float* dt_c, float* phi, float* st_re, float* st_im,
                       cudaStream_t s, void* re_bf, void* im_bf) {
  const bool tc_scan = re_bf && im_bf && scan_tc_supported(p);
  __nv_bfloat16* rb = tc_scan ? static_cast<__nv_bfloat16*>(re_bf) : nullptr;
  __nv_bfloat16* ib = tc_scan ? static_cast<__nv_bfloat16*>(im_bf) : nullptr;
  cudaError_t e = launch_chunk_cumsum(p, dA_cs, dt_c, s, phi);
  if (e != cudaSuccess) return e;
  const bool bf = p.io == SSD_DTYPE_BF16;
#define SSD_ROT_STATES(QQ)                                                                                   \
  if (bf) {                                                                                                  \
    if ((e = launch_state_t<__nv_bfloat16, QQ, kRotRe>(p, p.x, p.Bm, dA_cs, dt_c, phi, st_re, s)) != cudaSuccess) \
      return e;                                                                                              \
    if ((e = launch_state_t<__nv_bfloat16, QQ, kRotIm>(p, p.x, p.Bm, dA_cs, dt_c, phi, st_im, s)) != cudaSuccess) \
      return e;                                                                                              \
  } else {                                                                                                   \
    if ((e = launch_state_t<float, QQ, kRotRe>(p, p.x, p.Bm, dA_cs, dt_c, phi, st_re, s)) != cudaSuccess)  \
      return e;                                                                                              \
    if ((e = launch_state_t<float, QQ, kRotIm>(p, p.x, p.Bm, dA_cs, dt_c, phi, st_im, s)) != cudaSuccess)  \
      return e;                                                                                              \
  }
  if (use_state_tc(p)) {
    if ((e = launch_chunk_state_tc(p, kRotRe, p.x, p.Bm, dA_cs, dt_c, phi, st_re, s)) != cudaSuccess) return e;
    if ((e = launch_chunk_state_tc(p, kRotIm, p.x, p.Bm, dA_cs, dt_c, phi, st_im, s)) != cudaSuccess) return e;
  } else switch (p.Q) {
    case 32: SSD_ROT_STATES(32) break;
    case 64: SSD_ROT_STATES(64) break;
    case 128: SSD_ROT_STATES(128) break;
    default: return cudaErrorInvalidValue;
  }
#undef SSD_ROT_STATES
  {
    const int64_t PN = p.P * p.N;
    dim3 grid((unsigned)((PN + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.B);
    if (PN % 4 == 0) {
      dim3 g4((unsigned)((PN / 4 + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.B);
      state_passing_rot_kernel<4><<<g4, kThreads, 0, s>>>(dA_cs, phi, p.init, p.init_im, st_re, st_im,
                                                          p.final_state, p.final_im, p.H, PN, p.nc, (int)p.Q, rb, ib);
    } else {
      state_passing_rot_kernel<1><<<grid, kThreads, 0, s>>>(dA_cs, phi, p.init, p.init_im, st_re, st_im,
                                                            p.final_state, p.final_im, p.H, PN, p.nc, (int)p.Q, rb,
                                                            ib);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (tc_scan) return launch_chunk_scan_tc(p, dA_cs, dt_c, phi, rb, ib, s);
  switch (p.Q) {
    case 32: return bf ? launch_scan_t<__nv_bfloat16, 32, true>(p, dA_cs, dt_c, st_re, phi, st_im, s)
                       : launch_scan_t<float, 32, true>(p, dA_cs, dt_c, st_re, phi, st_im, s);
    case 64: return bf ? launch_scan_t<__nv_bfloat16, 64, true>(p, dA_cs, dt_c, st_re, phi, st_im, s)
                       : launch_scan_t<float, 64, true>(p, dA_cs, dt_c, st_re, phi, st_im, s);
    case 128: return bf ? launch_scan_t<__nv_bfloat16, 128, true>(p, dA_cs, dt_c, st_re, phi, st_im, s)
                        : launch_scan_t<float, 128, true>(p, dA_cs, dt_c, st_re, phi, st_im, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_chunk_cumsum(const Problem& p, float* dA_cs, float* dt_c, cudaStream_t s, float* phi) {
  const int hpb = 8;
  dim3 grid((unsigned)p.nc, (unsigned)((p.H + hpb - 1) / hpb), (unsigned)p.B);
  switch (p.Q) {
    case 32: chunk_cumsum_kernel<32><<<grid, 32, 0, s>>>(p.dt, p.dt_bias, p.dt_softplus, p.A, p.theta, p.L, p.H, p.nc, hpb, dA_cs, dt_c, phi); break;
    case 64: chunk_cumsum_kernel<64><<<grid, 64, 0, s>>>(p.dt, p.dt_bias, p.dt_softplus, p.A, p.theta, p.L, p.H, p.nc, hpb, dA_cs, dt_c, phi); break;
    case 128: chunk_cumsum_kernel<128><<<grid, 128, 0, s>>>(p.dt, p.dt_bias, p.dt_softplus, p.A, p.theta, p.L, p.H, p.nc, hpb, dA_cs, dt_c, phi); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_chunk_state(const Problem& p, const float* dA_cs, const float* dt_c,
                               float* states, cudaStream_t s) {
  if (use_state_tc(p)) return launch_chunk_state_tc(p, kFwd, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s);
  const bool bf = p.io == SSD_DTYPE_BF16;
  switch (p.Q) {
    case 32: return bf ? launch_state_t<__nv_bfloat16, 32, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s)
                       : launch_state_t<float, 32, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s);
    case 64: return bf ? launch_state_t<__nv_bfloat16, 64, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s)
                       : launch_state_t<float, 64, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s);
    case 128: return bf ? launch_state_t<__nv_bfloat16, 128, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s)
                        : launch_state_t<float, 128, kFwd>(p, p.x, p.Bm, dA_cs, dt_c, nullptr, states, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_chunk_state_adjoint(const Problem& p, const void* dy, const float* dA_cs,
                                       float* gstates, cudaStream_t s) {
  if (use_state_tc(p)) return launch_chunk_state_tc(p, kAdjoint, dy, p.Cm, dA_cs, nullptr, nullptr, gstates, s);
  const bool bf = p.io == SSD_DTYPE_BF16;
  switch (p.Q) {
    case 64: return bf ? launch_state_t<__nv_bfloat16, 64, kAdjoint>(p, dy, p.Cm, dA_cs, nullptr, nullptr, gstates, s)
                       : launch_state_t<float, 64, kAdjoint>(p, dy, p.Cm, dA_cs, nullptr, nullptr, gstates, s);
    case 128: return bf ? launch_state_t<__nv_bfloat16, 128, kAdjoint>(p, dy, p.Cm, dA_cs, nullptr, nullptr, gstates, s)
                        : launch_state_t<float, 128, kAdjoint>(p, dy, p.Cm, dA_cs, nullptr, nullptr, gstates, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_state_passing(const Problem& p, const float* dA_cs, float* states,
                                 cudaStream_t s, void* states_bf) {
  const int64_t PN = p.P * p.N;
  dim3 grid((unsigned)((PN + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.B);
  if (PN % 4 == 0) {
    dim3 g4((unsigned)((PN / 4 + kThreads - 1) / kThreads), (unsigned)p.H, (unsigned)p.B);
    state_passing_kernel<4><<<g4, kThreads, 0, s>>>(dA_cs, p.init, states, p.final_state, p.H, PN, p.nc, (int)p.Q,
                                                    static_cast<__nv_bfloat16*>(states_bf));
  } else {
    state_passing_kernel<1><<<grid, kThreads, 0, s>>>(dA_cs, p.init, states, p.final_state, p.H, PN, p.nc,
                                                      (int)p.Q, static_cast<__nv_bfloat16*>(states_bf));
  }
  return cudaGetLastError();
}

cudaError_t launch_chunk_scan(const Problem& p, const float* dA_cs, const float* dt_c,
                              const float* states, cudaStream_t s) {
  const bool bf = p.io == SSD_DTYPE_BF16;
  switch (p.Q) {
    case 32: return bf ? launch_scan_t<__nv_bfloat16, 32, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s)
                       : launch_scan_t<float, 32, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s);
    case 64: return bf ? launch_scan_t<__nv_bfloat16, 64, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s)
                       : launch_scan_t<float, 64, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s);
    case 128: return bf ? launch_scan_t<__nv_bfloat16, 128, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s)
                        : launch_scan_t<float, 128, false>(p, dA_cs, dt_c, states, nullptr, nullptr, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
