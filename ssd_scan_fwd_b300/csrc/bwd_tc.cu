// bwd_tc.cu -- the per-chunk gradients of the backward pass on the tensor
// cores (bf16 io, headdim 64, dstate 128, chunk 128).
//
// Same quantities as bwd_chunk_kernel in bwd.cu (the reverse-mode gradient
// of the recurrence of "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进", §2.1.2,
// written out there), for chunk c of head h with token rows t, s, j = 0..127:
//   DX = dY Xᵀ, CB = C Bᵀ (and their transposes), the mask E[s][j] =
//   e^{cs_s − cs_j} (s ≥ j),
//   M1ᵀ[t][s] = E[s][t] CB[s][t],  M2ᵀ[t][s] = E[s][t] DX[s][t],
//   M3[s][j]  = E[s][j] Δ_j DX[s][j],
//   u   = M1ᵀ dY + diag(e^{cs_last − cs}) B Goutᵀ,     dx = D dy + diag(Δ) u
//   dB  = diag(Δ) (M2ᵀ C + X̃ Gout),  X̃ = diag(e^{cs_last − cs}) X
//   dC  = M3 B + Ỹ Hin,                Ỹ = diag(e^{cs}) dY
//   the strict row and column sums of W = M3 ⊙ CB, and for dΔ, dA the
//   read-out terms e^{cs} C·(Hinᵀ dy) and Δ e^{cs_last − cs} x·(Gout B).
//
// One CTA of 128 threads per (chunk, head, batch row); thread r owns token
// row r, which is TMEM lane r of every accumulator.  TMA brings X, dY, B, C;
// the threads write X̃, Ỹ and bf16 copies of Gout and Hin (the fp32 states
// entering and leaving the chunk).  Stage 1: four SS MMAs (DX, CB, DXᵀ, CBᵀ:
// all 512 TMEM columns); each thread turns its rows into the masks M3, M1ᵀ,
// M2ᵀ as bf16 A operands written over the columns it has read.  Stage 2: u
// (TMEM A = M1ᵀ), Goutᵀ B, C Hinᵀ and dB (TMEM A = M2ᵀ plus X̃ Gout).  Stage 3:
// dC (TMEM A = M3 plus Ỹ Hin).  dB and dC are group sums: added to fp32
// accumulators with 16-byte atomics.  Waits are bounded (2 s).

#include <cuda.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "sm100.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQt = 128, kPt = 64, kNt = 128, kThr = 128;
constexpr uint32_t kBlk = kQt * 128;     // [128 rows][128 B]
constexpr uint32_t kBlkS = kPt * 128;    // [64 rows][128 B]
constexpr uint32_t kOX = 0;              // X  [t][p]
constexpr uint32_t kODY = kBlk;          // dY [t][p]
constexpr uint32_t kOB = 2 * kBlk;       // B  [t][n]: n 0-63, 64-127
constexpr uint32_t kOC = 4 * kBlk;       // C  [t][n]
constexpr uint32_t kOXS = 6 * kBlk;      // X̃ = diag(e^{cs_last - cs}) X
constexpr uint32_t kODYS = 7 * kBlk;     // Ỹ = diag(e^{cs}) dY
constexpr uint32_t kOG = 8 * kBlk;       // Gout (bf16) [p][n]: n 0-63, 64-127
constexpr uint32_t kOH = kOG + 2 * kBlkS;  // Hin (bf16) [p][n]
constexpr uint32_t kOV = kOH + 2 * kBlkS;  // vectors (fp32)
enum : int { V_CS = 0, V_DL = 128, V_WT = 256, V_COUNT = 256 + 4 * 8 };  // V_WT: per-warp totals
constexpr uint32_t kOBar = kOV + V_COUNT * 4;
constexpr uint32_t kOMisc = kOBar + 4 * 8;
constexpr uint32_t kSmem = kOMisc + 16 + 1024;
static_assert(kSmem <= 232448, "shared memory budget");

// TMEM columns
constexpr uint32_t T_DX = 0, T_CB = 128, T_DXT = 256, T_CBT = 384;  // stage 1
constexpr uint32_t T_M3 = 0, T_M2T = 256, T_M1T = 384;              // masks (bf16 pairs) over them
constexpr uint32_t T_U = 64, T_GB = 320, T_CH = 448, T_DB = 128;    // stage 2
constexpr uint32_t T_DC = 64;                                       // stage 3

constexpr uint32_t kIdSS128 = idesc_bf16_f32(128, 128, 0, 0);  // K-major · K-major, N = 128
constexpr uint32_t kIdSS64 = idesc_bf16_f32(128, 64, 0, 0);    // K-major · K-major, N = 64
constexpr uint32_t kIdMN128 = idesc_bf16_f32(128, 128, 0, 1);  // (TMEM or K-major) · MN-major, N = 128
constexpr uint32_t kIdMN64 = idesc_bf16_f32(128, 64, 0, 1);    // (TMEM or K-major) · MN-major, N = 64

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 2000000000ull) return false;
  }
  return true;
}

// K-major operand with K spread over 64-element column blocks of `blk` bytes:
// start-address step (16-byte units) of K step kk (16 elements).
__device__ __forceinline__ uint64_t kstep_cols(uint32_t kk, uint32_t blk) {
  return (uint64_t)((kk >> 2) * (blk >> 4) + (kk & 3u) * 2u);
}

struct BwdTcArgs {
  const float* A;
  const float* D;
  const float* dA_cs;
  const float* dt_c;
  const float* states;   // h_in per chunk [B][nc][H][P][N]
  const float* gstates;  // Gout per chunk
  void* dx;
  float* ddt;
  float* dB_acc;
  float* dC_acc;
  float* dA;
  float* dD;
  int64_t L, H, nc;
  int G;
};

__global__ void __launch_bounds__(kThr, 1)
    bwd_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                        const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                        const BwdTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  float* vec = reinterpret_cast<float*>(gbase + kOV);
  const uint32_t bar_load = sbase + kOBar, bar_m1 = bar_load + 8, bar_m2 = bar_load + 16, bar_m3 = bar_load + 24;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kOMisc);

  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = (int)(h / (a.H / a.G));
  const int r = threadIdx.x, warp = r >> 5;
  const uint32_t lane_addr = (32u * (uint32_t)warp) << 16;
  const int64_t t0 = c * kQt;

  if (r == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_m1, 1);
    mbar_init(bar_m2, 1);
    mbar_init(bar_m3, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + kOMisc, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (r == 0) {
    mbar_arrive_expect_tx(bar_load, 6 * kBlk);
    tma_load_3d(sbase + kOX, &tm_x, bar_load, (int32_t)(h * kPt), (int32_t)t0, (int32_t)b);
    tma_load_3d(sbase + kODY, &tm_dy, bar_load, (int32_t)(h * kPt), (int32_t)t0, (int32_t)b);
    tma_load_3d(sbase + kOB, &tm_b, bar_load, g * kNt, (int32_t)t0, (int32_t)b);
    tma_load_3d(sbase + kOB + kBlk, &tm_b, bar_load, g * kNt + 64, (int32_t)t0, (int32_t)b);
    tma_load_3d(sbase + kOC, &tm_c, bar_load, g * kNt, (int32_t)t0, (int32_t)b);
    tma_load_3d(sbase + kOC + kBlk, &tm_c, bar_load, g * kNt + 64, (int32_t)t0, (int32_t)b);
  }
  // per-token scalars; bf16 copies of Gout and Hin (swizzled, [p][n] in two
  // 64-column blocks) and γ = <Gout, Hin>
  const int64_t vrow = ((b * a.H + h) * a.nc + c) * kQt;
  vec[V_CS + r] = a.dA_cs[vrow + r];
  vec[V_DL + r] = a.dt_c[vrow + r];
  float gam = 0.f;
  {
    const int64_t srow = ((b * a.nc + c) * a.H + h) * (int64_t)kPt * kNt;
    const float* gout = a.gstates + srow;
    const float* hin = a.states + srow;
    for (int e = r; e < kPt * 16; e += kThr) {  // (p, 8-column chunk): 64 rows × 16 chunks
      const int p = e >> 4, k = e & 15, blk = k >> 3, ch = k & 7;
      const float4* gs = reinterpret_cast<const float4*>(gout + (int64_t)p * kNt + 8 * k);
      const float4* hs = reinterpret_cast<const float4*>(hin + (int64_t)p * kNt + 8 * k);
      const float4 g0 = gs[0], g1 = gs[1], h0 = hs[0], h1 = hs[1];
      gam += g0.x * h0.x + g0.y * h0.y + g0.z * h0.z + g0.w * h0.w + g1.x * h1.x + g1.y * h1.y + g1.z * h1.z +
             g1.w * h1.w;
      const uint32_t off = (uint32_t)blk * kBlkS + sw128_offset((uint32_t)p, (uint32_t)ch);
      *reinterpret_cast<uint4*>(gbase + kOG + off) =
          make_uint4(pack_bf16x2(g0.x, g0.y), pack_bf16x2(g0.z, g0.w), pack_bf16x2(g1.x, g1.y), pack_bf16x2(g1.z, g1.w));
      *reinterpret_cast<uint4*>(gbase + kOH + off) =
          make_uint4(pack_bf16x2(h0.x, h0.y), pack_bf16x2(h0.z, h0.w), pack_bf16x2(h1.x, h1.y), pack_bf16x2(h1.z, h1.w));
    }
  }
  bool ok = __syncthreads_and(wait_bounded(bar_load, 0));
  const float cs_last = vec[V_CS + kQt - 1];
  const float cs_r = vec[V_CS + r], dl_r = vec[V_DL + r];
  if (ok) {
    // X̃ and Ỹ: row r scaled
    const uint32_t wx = pack_bf16x2(expf(cs_last - cs_r), expf(cs_last - cs_r));
    const uint32_t wy = pack_bf16x2(expf(cs_r), expf(cs_r));
#pragma unroll
    for (uint32_t ch = 0; ch < 8; ++ch) {
      const uint32_t off = sw128_offset((uint32_t)r, ch);
      uint4 v = *reinterpret_cast<const uint4*>(gbase + kOX + off);
      v.x = mul_bf16x2(v.x, wx);
      v.y = mul_bf16x2(v.y, wx);
      v.z = mul_bf16x2(v.z, wx);
      v.w = mul_bf16x2(v.w, wx);
      *reinterpret_cast<uint4*>(gbase + kOXS + off) = v;
      uint4 u = *reinterpret_cast<const uint4*>(gbase + kODY + off);
      u.x = mul_bf16x2(u.x, wy);
      u.y = mul_bf16x2(u.y, wy);
      u.z = mul_bf16x2(u.z, wy);
      u.w = mul_bf16x2(u.w, wy);
      *reinterpret_cast<uint4*>(gbase + kODYS + off) = u;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ---- stage 1: DX = dY Xᵀ, CB = C Bᵀ, DXᵀ = X dYᵀ, CBᵀ = B Cᵀ
  if (ok && r == 0) {
    tc_fence_after();
    const uint64_t dX = smem_desc_sw128(sbase + kOX, 16, 1024), dDY = smem_desc_sw128(sbase + kODY, 16, 1024);
    const uint64_t dB = smem_desc_sw128(sbase + kOB, 16, 1024), dC = smem_desc_sw128(sbase + kOC, 16, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < 4; ++kk) {
      mma_ss(tmem + T_DX, dDY + kk * 2u, dX + kk * 2u, kIdSS128, kk > 0);
      mma_ss(tmem + T_DXT, dX + kk * 2u, dDY + kk * 2u, kIdSS128, kk > 0);
    }
#pragma unroll
    for (uint32_t kk = 0; kk < 8; ++kk) {
      mma_ss(tmem + T_CB, dC + kstep_cols(kk, kBlk), dB + kstep_cols(kk, kBlk), kIdSS128, kk > 0);
      mma_ss(tmem + T_CBT, dB + kstep_cols(kk, kBlk), dC + kstep_cols(kk, kBlk), kIdSS128, kk > 0);
    }
    mma_commit(bar_m1);
  }
  if (ok) ok = wait_bounded(bar_m1, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  float rowsum = 0.f, colsum = 0.f, dd = 0.f;
  if (ok) {
    // row s = r of DX, CB: M3 and the strict row sum of W; the trace of DX
#pragma unroll 1
    for (uint32_t jc = 0; jc < 4; ++jc) {
      uint32_t dxr[32], cbr[32];
      tmem_ld32(tmem + lane_addr + T_DX + 32u * jc, dxr);
      tmem_ld32(tmem + lane_addr + T_CB + 32u * jc, cbr);
      tmem_ld_wait();
      reg_fence(dxr);
      reg_fence(cbr);
      uint32_t m3[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float w2[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int j = 32 * (int)jc + e + q;
          const float dxv = __uint_as_float(dxr[e + q]);
          const float E = j <= r ? expf(cs_r - vec[V_CS + j]) : 0.f;
          const float wc = E * vec[V_DL + j] * dxv;
          if (j < r) rowsum = fmaf(wc, __uint_as_float(cbr[e + q]), rowsum);
          if (j == r) dd += dxv;
          w2[q] = wc;
        }
        m3[e >> 1] = pack_bf16x2(w2[0], w2[1]);
      }
      tmem_st16(tmem + lane_addr + T_M3 + 16u * jc, m3);
    }
    // row t = r of DXᵀ, CBᵀ: M1ᵀ, M2ᵀ and the strict column sum of W
#pragma unroll 1
    for (uint32_t sc = 0; sc < 4; ++sc) {
      uint32_t dxt[32], cbt[32];
      tmem_ld32(tmem + lane_addr + T_DXT + 32u * sc, dxt);
      tmem_ld32(tmem + lane_addr + T_CBT + 32u * sc, cbt);
      tmem_ld_wait();
      reg_fence(dxt);
      reg_fence(cbt);
      uint32_t m1[16], m2[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float a1v[2], a2v[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int s = 32 * (int)sc + e + q;
          const float E = s >= r ? expf(vec[V_CS + s] - cs_r) : 0.f;
          const float dxv = __uint_as_float(dxt[e + q]), cbv = __uint_as_float(cbt[e + q]);
          a1v[q] = E * cbv;
          a2v[q] = E * dxv;
          if (s > r) colsum = fmaf(E * dxv, cbv, colsum);
        }
        m1[e >> 1] = pack_bf16x2(a1v[0], a1v[1]);
        m2[e >> 1] = pack_bf16x2(a2v[0], a2v[1]);
      }
      tmem_st16(tmem + lane_addr + T_M1T + 16u * sc, m1);
      tmem_st16(tmem + lane_addr + T_M2T + 16u * sc, m2);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();

  // ---- stage 2: u (M1ᵀ dY), GB = B Goutᵀ, CH = C Hinᵀ, dB (M2ᵀ C + X̃ Gout)
  if (ok && r == 0) {
    tc_fence_after();
    const uint64_t dDYm = smem_desc_sw128(sbase + kODY, kBlk, 1024);   // dY [s][p] MN-major
    const uint64_t dB = smem_desc_sw128(sbase + kOB, 16, 1024), dC = smem_desc_sw128(sbase + kOC, 16, 1024);
    const uint64_t dG = smem_desc_sw128(sbase + kOG, 16, 1024), dH = smem_desc_sw128(sbase + kOH, 16, 1024);
    const uint64_t dCm = smem_desc_sw128(sbase + kOC, kBlk, 1024);     // C [s][n] MN-major
    const uint64_t dGm = smem_desc_sw128(sbase + kOG, kBlkS, 1024);    // Gout [p][n] MN-major
    const uint64_t dXS = smem_desc_sw128(sbase + kOXS, 16, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < 8; ++kk) {
      mma_ts(tmem + T_U, tmem + T_M1T + kk * 8u, dDYm + kk * 128u, kIdMN64, kk > 0);
      mma_ss(tmem + T_GB, dB + kstep_cols(kk, kBlk), dG + kstep_cols(kk, kBlkS), kIdSS64, kk > 0);
      mma_ss(tmem + T_CH, dC + kstep_cols(kk, kBlk), dH + kstep_cols(kk, kBlkS), kIdSS64, kk > 0);
      mma_ts(tmem + T_DB, tmem + T_M2T + kk * 8u, dCm + kk * 128u, kIdMN128, kk > 0);
    }
#pragma unroll
    for (uint32_t kk = 0; kk < 4; ++kk) mma_ss(tmem + T_DB, dXS + kk * 2u, dGm + kk * 128u, kIdMN128, 1);
    mma_commit(bar_m2);
  }
  if (ok) ok = wait_bounded(bar_m2, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  const int64_t tt = t0 + r;
  const bool live = tt < a.L;
  const float eg = expf(cs_last - cs_r), ecs = expf(cs_r);
  float xu = 0.f, gbx = 0.f, a1 = 0.f;
  if (ok) {
    const float Dh = a.D ? a.D[h] : 0.f;
#pragma unroll 1
    for (uint32_t hp = 0; hp < 2; ++hp) {
      uint32_t ur[32], gr[32], cr[32];
      tmem_ld32(tmem + lane_addr + T_U + 32u * hp, ur);
      tmem_ld32(tmem + lane_addr + T_GB + 32u * hp, gr);
      tmem_ld32(tmem + lane_addr + T_CH + 32u * hp, cr);
      tmem_ld_wait();
      reg_fence(ur);
      reg_fence(gr);
      reg_fence(cr);
      uint32_t dxo[16];
#pragma unroll
      for (uint32_t ch = 0; ch < 4; ++ch) {
        const uint32_t off = sw128_offset((uint32_t)r, 4 * hp + ch);
        const uint4 xv = *reinterpret_cast<const uint4*>(gbase + kOX + off);
        const uint4 yv = *reinterpret_cast<const uint4*>(gbase + kODY + off);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, yw[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 8 * (int)ch + 2 * q;
          const float x0 = bf16lo_to_f(xw[q]), x1 = bf16hi_to_f(xw[q]);
          const float y0 = bf16lo_to_f(yw[q]), y1 = bf16hi_to_f(yw[q]);
          const float g0 = __uint_as_float(gr[e]), g1 = __uint_as_float(gr[e + 1]);
          const float u0 = fmaf(eg, g0, __uint_as_float(ur[e])), u1 = fmaf(eg, g1, __uint_as_float(ur[e + 1]));
          xu = fmaf(x0, u0, fmaf(x1, u1, xu));
          gbx = fmaf(x0, g0, fmaf(x1, g1, gbx));
          a1 = fmaf(y0, __uint_as_float(cr[e]), fmaf(y1, __uint_as_float(cr[e + 1]), a1));
          dxo[e >> 1] = pack_bf16x2(fmaf(Dh, y0, dl_r * u0), fmaf(Dh, y1, dl_r * u1));
        }
      }
      if (live) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.dx) + ((b * a.L + tt) * a.H + h) * kPt +
                                              32 * hp);
#pragma unroll
        for (int q = 0; q < 4; ++q) dst[q] = make_uint4(dxo[4 * q], dxo[4 * q + 1], dxo[4 * q + 2], dxo[4 * q + 3]);
      }
    }
    // dB row: Δ_t (M2ᵀ C + X̃ Gout)
#pragma unroll 1
    for (uint32_t nq = 0; nq < 4; ++nq) {
      uint32_t br[32];
      tmem_ld32(tmem + lane_addr + T_DB + 32u * nq, br);
      tmem_ld_wait();
      reg_fence(br);
      if (live) {
        float4* dst = reinterpret_cast<float4*>(a.dB_acc + ((b * a.L + tt) * a.G + g) * kNt + 32 * nq);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          atomicAdd(dst + q, make_float4(dl_r * __uint_as_float(br[4 * q]), dl_r * __uint_as_float(br[4 * q + 1]),
                                         dl_r * __uint_as_float(br[4 * q + 2]), dl_r * __uint_as_float(br[4 * q + 3])));
      }
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- stage 3: dC = M3 B + Ỹ Hin
  if (ok && r == 0) {
    tc_fence_after();
    const uint64_t dBm = smem_desc_sw128(sbase + kOB, kBlk, 1024);   // B [j][n] MN-major
    const uint64_t dHm = smem_desc_sw128(sbase + kOH, kBlkS, 1024);  // Hin [p][n] MN-major
    const uint64_t dYS = smem_desc_sw128(sbase + kODYS, 16, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < 8; ++kk) mma_ts(tmem + T_DC, tmem + T_M3 + kk * 8u, dBm + kk * 128u, kIdMN128, kk > 0);
#pragma unroll
    for (uint32_t kk = 0; kk < 4; ++kk) mma_ss(tmem + T_DC, dYS + kk * 2u, dHm + kk * 128u, kIdMN128, 1);
    mma_commit(bar_m3);
  }
  if (ok) ok = wait_bounded(bar_m3, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
#pragma unroll 1
    for (uint32_t nq = 0; nq < 4; ++nq) {
      uint32_t cr[32];
      tmem_ld32(tmem + lane_addr + T_DC + 32u * nq, cr);
      tmem_ld_wait();
      reg_fence(cr);
      if (live) {
        float4* dst = reinterpret_cast<float4*>(a.dC_acc + ((b * a.L + tt) * a.G + g) * kNt + 32 * nq);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          atomicAdd(dst + q, make_float4(__uint_as_float(cr[4 * q]), __uint_as_float(cr[4 * q + 1]),
                                         __uint_as_float(cr[4 * q + 2]), __uint_as_float(cr[4 * q + 3])));
      }
    }
  }
  tc_fence_before();
  // dΔ, dA, dD.  Per token k (all terms of thread k):
  //   da_k = Σ_{i<k} (cols_i − rows_i) + Σ_{s≥k} e^{cs_s} C_s·(Hinᵀ dy_s)
  //        + Σ_{j<k} Δ_j e^{cs_last − cs_j} x_j·(Gout B_j) + e^{cs_last} <Gout, Hin>
  // as block scans: inclusive warp scans, then the warps' totals.
  const int lane = r & 31;
  const float v1 = dl_r * colsum - rowsum, v2 = ecs * a1, v3 = dl_r * eg * gbx;
  float s1 = v1, s2 = v2, s3 = v3, sg = gam, sd = dd;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float t1 = __shfl_up_sync(0xffffffffu, s1, off), t2 = __shfl_up_sync(0xffffffffu, s2, off),
                t3 = __shfl_up_sync(0xffffffffu, s3, off);
    if (lane >= off) {
      s1 += t1;
      s2 += t2;
      s3 += t3;
    }
    sg += __shfl_xor_sync(0xffffffffu, sg, off);
    sd += __shfl_xor_sync(0xffffffffu, sd, off);
  }
  if (lane == 31) {
    vec[V_WT + 8 * warp + 0] = s1;
    vec[V_WT + 8 * warp + 1] = s2;
    vec[V_WT + 8 * warp + 2] = s3;
    vec[V_WT + 8 * warp + 3] = sg;
    vec[V_WT + 8 * warp + 4] = sd;
  }
  __syncthreads();
  float o1 = 0.f, o2 = 0.f, o3 = 0.f, tot2 = 0.f, gsum = 0.f, dsum = 0.f;
#pragma unroll
  for (int w = 0; w < kThr / 32; ++w) {
    if (w < warp) {
      o1 += vec[V_WT + 8 * w + 0];
      o2 += vec[V_WT + 8 * w + 1];
      o3 += vec[V_WT + 8 * w + 2];
    }
    tot2 += vec[V_WT + 8 * w + 1];
    gsum += vec[V_WT + 8 * w + 3];
    dsum += vec[V_WT + 8 * w + 4];
  }
  const float da = (s1 - v1 + o1) + (tot2 - (s2 + o2) + v2) + (s3 - v3 + o3) + expf(cs_last) * gsum;
  if (ok && live) a.ddt[(b * a.L + tt) * a.H + h] = fmaf(a.A[h], da, xu);
  float dAp = dl_r * da;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) dAp += __shfl_xor_sync(0xffffffffu, dAp, off);
  __syncthreads();
  if (lane == 0) vec[V_WT + 8 * warp + 5] = dAp;
  __syncthreads();
  if (ok && r == 0) {
    float dAsum = 0.f;
    for (int w = 0; w < kThr / 32; ++w) dAsum += vec[V_WT + 8 * w + 5];
    atomicAdd(a.dA + h, dAsum);
    if (a.D && a.dD) atomicAdd(a.dD + h, dsum);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool bwd_tc_supported(const Problem& p) {
  return p.io == SSD_DTYPE_BF16 && p.P == kPt && p.N == kNt && p.B > 0 && p.L > 0;
}

cudaError_t launch_bwd_chunk_tc(const BwdProblem& q, const float* dA_cs, const float* dt_c, const float* states,
                                const float* gstates, float* dB_acc, float* dC_acc, cudaStream_t s) {
  const Problem& p = q.fwd;
  if (!bwd_tc_supported(p) || p.Q != kQt) return cudaErrorNotSupported;
  CUtensorMap tx, tdy, tb, tc;
  if (!make_tma_map_bf16(&tx, p.x, p.B, p.L, p.H * kPt, kQt) ||
      !make_tma_map_bf16(&tdy, q.dy, p.B, p.L, p.H * kPt, kQt) ||
      !make_tma_map_bf16(&tb, p.Bm, p.B, p.L, p.G * kNt, kQt) ||
      !make_tma_map_bf16(&tc, p.Cm, p.B, p.L, p.G * kNt, kQt))
    return cudaErrorInvalidValue;
  BwdTcArgs a;
  a.A = p.A;
  a.D = p.D;
  a.dA_cs = dA_cs;
  a.dt_c = dt_c;
  a.states = states;
  a.gstates = gstates;
  a.dx = q.dx;
  a.ddt = q.ddt;
  a.dB_acc = dB_acc;
  a.dC_acc = dC_acc;
  a.dA = q.dA;
  a.dD = q.dD;
  a.L = p.L;
  a.H = p.H;
  a.nc = p.nc;
  a.G = (int)p.G;
  cudaError_t e = cudaFuncSetAttribute(bwd_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
  bwd_chunk_tc_kernel<<<grid, kThr, kSmem, s>>>(tx, tdy, tb, tc, a);
  return cudaGetLastError();
}

}  // namespace ssd
