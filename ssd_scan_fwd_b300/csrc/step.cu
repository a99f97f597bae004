// step.cu -- one recurrent step of the selective SSM per (batch row, head),
// the inference mode of the same recurrence the chunked forward pass
// evaluates ("Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of SSM)":
// the boxed recurrence of §2.1.2, h_t = α_t h_{t-1} + Δ_t B_t x_t with
// α_t = e^{Δ_t A}, read out as y_t = C_tᵀ h_t, plus the skip term D x of
// §2.1.1; §2.2.2: at inference the dual form switches back to this
// recurrence, with an O(1) state per head).
//
// The state is read and written once per call: the step is bound by HBM on
// the state (2 · P · N · 4 bytes per head).  One CTA per (b, h); each warp
// owns rows p of the state and walks n with 16-byte vectors, so a warp reads
// and writes whole 512-byte row segments, four rows at a time so that enough
// loads are in flight to cover the memory latency.

#include <cuda_bf16.h>

#include "internal.h"

namespace ssd {
namespace {

constexpr int kStepThreads = 256;

__device__ __forceinline__ float ld_io(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_io(const __nv_bfloat16* p, int64_t i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ void st_io(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_io(__nv_bfloat16* p, int64_t i, float v) { p[i] = __float2bfloat16_rn(v); }

struct StepParams {
  const void* x;
  const float* dt;
  const float* A;
  const void* Bm;
  const void* Cm;
  const float* D;
  float* state;
  void* y;
  int32_t H, P, G, N;
};

// VEC = 4: state rows are 16-byte aligned (N a multiple of 4); VEC = 1 otherwise.
template <typename T, int VEC>
__global__ void __launch_bounds__(kStepThreads) ssd_step_kernel(const StepParams p) {
  const int64_t bh = blockIdx.x;
  const int b = (int)(bh / p.H), h = (int)(bh % p.H);
  const int g = h / (p.H / p.G);
  const float dt = p.dt[bh];
  const float alpha = expf(dt * p.A[h]);
  const float Dh = p.D ? p.D[h] : 0.f;
  const T* x = static_cast<const T*>(p.x) + bh * p.P;
  const T* Bv = static_cast<const T*>(p.Bm) + ((int64_t)b * p.G + g) * p.N;
  const T* Cv = static_cast<const T*>(p.Cm) + ((int64_t)b * p.G + g) * p.N;
  T* y = static_cast<T*>(p.y) + bh * p.P;
  float* st = p.state + bh * (int64_t)p.P * p.N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kWarps = kStepThreads / 32;
  constexpr int kRows = 4;  // state rows per warp in flight (16-byte loads issued before use)
  for (int p0 = warp; p0 < p.P; p0 += kWarps * kRows) {
    float xv[kRows], acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const int pp = p0 + r * kWarps;
      xv[r] = pp < p.P ? ld_io(x, pp) : 0.f;
      acc[r] = 0.f;
    }
    for (int n0 = lane * VEC; n0 < p.N; n0 += 32 * VEC) {
      if constexpr (VEC == 4) {
        float4 hv[kRows];
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const int pp = p0 + r * kWarps;
          if (pp < p.P) hv[r] = *reinterpret_cast<const float4*>(st + (int64_t)pp * p.N + n0);
        }
        const float b0 = ld_io(Bv, n0), b1 = ld_io(Bv, n0 + 1), b2 = ld_io(Bv, n0 + 2), b3 = ld_io(Bv, n0 + 3);
        const float c0 = ld_io(Cv, n0), c1 = ld_io(Cv, n0 + 1), c2 = ld_io(Cv, n0 + 2), c3 = ld_io(Cv, n0 + 3);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const int pp = p0 + r * kWarps;
          if (pp >= p.P) continue;
          const float dx = dt * xv[r];
          float4 h = hv[r];
          h.x = fmaf(alpha, h.x, dx * b0);
          h.y = fmaf(alpha, h.y, dx * b1);
          h.z = fmaf(alpha, h.z, dx * b2);
          h.w = fmaf(alpha, h.w, dx * b3);
          acc[r] = fmaf(c0, h.x, acc[r]);
          acc[r] = fmaf(c1, h.y, acc[r]);
          acc[r] = fmaf(c2, h.z, acc[r]);
          acc[r] = fmaf(c3, h.w, acc[r]);
          *reinterpret_cast<float4*>(st + (int64_t)pp * p.N + n0) = h;
        }
      } else {
        const float bn = ld_io(Bv, n0), cn = ld_io(Cv, n0);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
          const int pp = p0 + r * kWarps;
          if (pp >= p.P) continue;
          float* row = st + (int64_t)pp * p.N;
          const float hv = fmaf(alpha, row[n0], dt * xv[r] * bn);
          acc[r] = fmaf(cn, hv, acc[r]);
          row[n0] = hv;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      float a = acc[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      const int pp = p0 + r * kWarps;
      if (lane == 0 && pp < p.P) st_io(y, pp, a + Dh * xv[r]);
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepProblem& q, cudaStream_t s) {
  if (q.B == 0) return cudaSuccess;
  StepParams sp;
  sp.x = q.x;
  sp.dt = q.dt;
  sp.A = q.A;
  sp.Bm = q.Bm;
  sp.Cm = q.Cm;
  sp.D = q.D;
  sp.state = q.state;
  sp.y = q.y;
  sp.H = (int32_t)q.H;
  sp.P = (int32_t)q.P;
  sp.G = (int32_t)q.G;
  sp.N = (int32_t)q.N;
  const unsigned grid = (unsigned)(q.B * q.H);
  const bool vec = (q.N % 4) == 0;
  if (q.io == SSD_DTYPE_BF16) {
    if (vec)
      ssd_step_kernel<__nv_bfloat16, 4><<<grid, kStepThreads, 0, s>>>(sp);
    else
      ssd_step_kernel<__nv_bfloat16, 1><<<grid, kStepThreads, 0, s>>>(sp);
  } else {
    if (vec)
      ssd_step_kernel<float, 4><<<grid, kStepThreads, 0, s>>>(sp);
    else
      ssd_step_kernel<float, 1><<<grid, kStepThreads, 0, s>>>(sp);
  }
  return cudaGetLastError();
}

}  // namespace ssd
