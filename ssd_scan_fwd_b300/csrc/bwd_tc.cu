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
//   read-out terms e^{cs} C·(Hinᵀ dy), Δ e^{cs_last − cs} x·(Gout B) and
//   e^{cs_last} <Gout, Hin>.
//
// One persistent CTA of 256 threads per SM walks the (chunk, head, batch row)
// items; the tiles of its next item are loaded while the current one
// finishes its atomics and scans.  Token row r is TMEM lane r of every
// accumulator; warps w and w + 4 share the lanes of quarter
// w mod 4, so each row has one thread in warpgroup 0 and one in warpgroup 1,
// which split the columns.  TMA brings X, dY, B, C and the bf16 copies of
// Gout and Hin (written by the two state recurrences); warpgroup 0 writes X̃,
// warpgroup 1 Ỹ.  Stage 1: four SS MMAs (DX, CB, DXᵀ, CBᵀ: all 512 TMEM
// columns); warpgroup 0 turns rows of DX, CB into M3 and the row sums of W,
// warpgroup 1 rows of DXᵀ, CBᵀ into M1ᵀ, M2ᵀ and the column sums, each as bf16
// A operands written over the columns it has read.  Column blocks wholly
// above (below) the diagonal are stored as zeros without being read.
// Stage 2: u (TMEM A = M1ᵀ), B Goutᵀ, C Hinᵀ (read by warpgroup 0: dx, and
// the dot products x·u, x·(Gout B), dy·(Hin C)) and dB (TMEM A = M2ᵀ, plus
// X̃ Gout; read by warpgroup 1).  Stage 3: dC (TMEM A = M3, plus Ỹ Hin), half
// the columns per warpgroup.  dB and dC are group sums: each item's rows are
// staged in shared memory (four [128 t][32 n] fp32 boxes, 64 KB) and added to
// the fp32 accumulators by TMA bulk reductions (cp.reduce.async.bulk .add,
// performed at L2), issued by thread 0; the staging is reused once the
// previous reduction has read it.  Exponentials are ex2 of the running sums
// prescaled by log2 e.  Waits are bounded (2 s).

#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "internal.h"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kQt = 128, kPt = 64, kNt = 128, kThr = 256;
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
constexpr uint32_t kOStg = kOH + 2 * kBlkS;  // dB / dC rows staged for the bulk reductions: 4 boxes [t][32 n] fp32
constexpr uint32_t kOV = kOStg + 4 * kBlk;   // vectors (fp32)
enum : int {
  V_CS2 = 0,        // cs · log2 e
  V_DL = 128,       // Δ
  V_COLS = 256,     // Δ_t Σ_{s>t} W[s][t] (warpgroup 1 -> 0)
  V_WT = 384,       // per-warp partial sums, 8 per warp
  V_COUNT = 384 + 8 * 8
};
constexpr uint32_t kOBar = kOV + V_COUNT * 4;
constexpr uint32_t kOMisc = kOBar + 6 * 8;
constexpr uint32_t kSmem = kOMisc + 16 + 1024;
constexpr uint32_t kLoadBytes = 6 * kBlk + 4 * kBlkS;
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

struct BwdTcArgs {
  const float* A;
  const float* D;
  const float* dA_cs;
  const float* dt_c;
  void* dx;
  float* ddt;
  float* dB_acc;
  float* dC_acc;
  float* dA;
  float* dD;
  int64_t B, L, H, nc;
  int G;
  int32_t* err;  // SSD_ERR_TIMEOUT is written here when a bounded wait gives up (may be null)
};

// Row pass over the 32 columns j = 32 jc .. of row s (warpgroup 0): M3 as
// bf16 pairs, Σ_{j<s} W[s][j] and DX[s][s].  kDiag: the block holding the
// diagonal (mask j ≤ s); otherwise every j < s.
template <bool kDiag>
__device__ __forceinline__ void row_block(const uint32_t (&dxr)[32], const uint32_t (&cbr)[32], const float* cs2,
                                          const float* dl, int jc, int s, float cs2_s, float& rowsum, float& dd,
                                          uint32_t (&m3)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float w2[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = 32 * jc + e + q;
      const float dxv = __uint_as_float(dxr[e + q]);
      float wc = ex2(cs2_s - cs2[j]) * dl[j] * dxv;
      if (kDiag) {
        if (j > s) wc = 0.f;
        if (j == s) dd = dxv;
        if (j < s) rowsum = fmaf(wc, __uint_as_float(cbr[e + q]), rowsum);
      } else {
        rowsum = fmaf(wc, __uint_as_float(cbr[e + q]), rowsum);
      }
      w2[q] = wc;
    }
    m3[e >> 1] = pack_bf16x2(w2[0], w2[1]);
  }
}

// Transposed pass over the 32 columns s = 32 sc .. of row t (warpgroup 1):
// M1ᵀ, M2ᵀ as bf16 pairs and Σ_{s>t} E[s][t] DX[s][t] CB[s][t].  kDiag: mask
// s ≥ t; otherwise every s > t.
template <bool kDiag>
__device__ __forceinline__ void col_block(const uint32_t (&dxt)[32], const uint32_t (&cbt)[32], const float* cs2,
                                          int sc, int t, float cs2_t, float& colsum, uint32_t (&m1)[16],
                                          uint32_t (&m2)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float a1v[2], a2v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int s = 32 * sc + e + q;
      float E = ex2(cs2[s] - cs2_t);
      if (kDiag && s < t) E = 0.f;
      const float dxv = __uint_as_float(dxt[e + q]), cbv = __uint_as_float(cbt[e + q]);
      a1v[q] = E * cbv;
      a2v[q] = E * dxv;
      if (!kDiag || s > t) colsum = fmaf(a2v[q], cbv, colsum);
    }
    m1[e >> 1] = pack_bf16x2(a1v[0], a1v[1]);
    m2[e >> 1] = pack_bf16x2(a2v[0], a2v[1]);
  }
}

__global__ void __launch_bounds__(kThr, 1)
    bwd_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_dy,
                        const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                        const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_h,
                        const __grid_constant__ CUtensorMap tm_db, const __grid_constant__ CUtensorMap tm_dc,
                        const BwdTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  float* vec = reinterpret_cast<float*>(gbase + kOV);
  const float* cs2 = vec + V_CS2;
  const float* dl = vec + V_DL;
  const uint32_t bar_load = sbase + kOBar, bar_m1 = bar_load + 8, bar_m2 = bar_load + 16, bar_m3 = bar_load + 24;
  const uint32_t bar_m2b = bar_load + 32;  // the dB MMAs of stage 2 (bar_m2: u, GB, CH)
  const uint32_t bar_m1b = bar_load + 40;  // DXᵀ, CBᵀ of stage 1 (bar_m1: DX, CB)
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kOMisc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2, quarter = warp & 3;
  const int r = 32 * quarter + lane;  // token row = TMEM lane
  const uint32_t lane_addr = (32u * (uint32_t)quarter) << 16;
  const int64_t n_items = a.nc * a.H * a.B;  // item k: chunk k mod nc, head (k / nc) mod H, batch row k / (nc H)

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_m1, 1);
    mbar_init(bar_m2, 1);
    mbar_init(bar_m3, 1);
    mbar_init(bar_m2b, 1);
    mbar_init(bar_m1b, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + kOMisc, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // TMA loads of item k (thread 0)
  auto issue_loads = [&](int64_t k) {
    const int64_t kc = k % a.nc, kh = (k / a.nc) % a.H, kb = k / (a.nc * a.H);
    const int kg = (int)(kh / (a.H / a.G));
    const int32_t kt0 = (int32_t)(kc * kQt);
    const int32_t srow = (int32_t)(((kb * a.nc + kc) * a.H + kh) * kPt);  // row of the [p][n] state slabs
    mbar_arrive_expect_tx(bar_load, kLoadBytes);
    tma_load_3d(sbase + kOX, &tm_x, bar_load, (int32_t)(kh * kPt), kt0, (int32_t)kb);
    tma_load_3d(sbase + kODY, &tm_dy, bar_load, (int32_t)(kh * kPt), kt0, (int32_t)kb);
    tma_load_3d(sbase + kOB, &tm_b, bar_load, kg * kNt, kt0, (int32_t)kb);
    tma_load_3d(sbase + kOB + kBlk, &tm_b, bar_load, kg * kNt + 64, kt0, (int32_t)kb);
    tma_load_3d(sbase + kOC, &tm_c, bar_load, kg * kNt, kt0, (int32_t)kb);
    tma_load_3d(sbase + kOC + kBlk, &tm_c, bar_load, kg * kNt + 64, kt0, (int32_t)kb);
    tma_load_3d(sbase + kOG, &tm_g, bar_load, 0, srow, 0);
    tma_load_3d(sbase + kOG + kBlkS, &tm_g, bar_load, 64, srow, 0);
    tma_load_3d(sbase + kOH, &tm_h, bar_load, 0, srow, 0);
    tma_load_3d(sbase + kOH + kBlkS, &tm_h, bar_load, 64, srow, 0);
  };
  if (tid == 0 && (int64_t)blockIdx.x < n_items) issue_loads(blockIdx.x);

  // Persistent loop over items; each barrier completes once per item.  The
  // next item's tiles are requested as soon as this item's last MMAs are
  // done, so they arrive while its dC atomics and scans run.
  bool ok = true;
  uint32_t ph = 0;
  for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x, ph ^= 1u) {
    const int64_t c = item % a.nc, h = (item / a.nc) % a.H, b = item / (a.nc * a.H);
    const int g = (int)(h / (a.H / a.G));
    const int64_t t0 = c * kQt;
    {
      const int64_t vrow = ((b * a.H + h) * a.nc + c) * kQt;
      if (wg == 0)
        vec[V_CS2 + r] = a.dA_cs[vrow + r] * kLog2e;
      else
        vec[V_DL + r] = a.dt_c[vrow + r];
    }
    ok = __syncthreads_and(wait_bounded(bar_load, ph));
    const float cs2_last = cs2[kQt - 1];
    const float cs2_r = cs2[r], dl_r = dl[r];
    float gam = 0.f;  // <Gout, Hin>: the two tiles share one layout, so pair them element by element
    if (ok) {
      // X̃ (warpgroup 0) or Ỹ (warpgroup 1): row r scaled
      const float wv = wg == 0 ? ex2(cs2_last - cs2_r) : ex2(cs2_r);
      const uint32_t w2 = pack_bf16x2(wv, wv);
      const uint32_t src = wg == 0 ? kOX : kODY, dst = wg == 0 ? kOXS : kODYS;
  #pragma unroll
      for (uint32_t ch = 0; ch < 8; ++ch) {
        const uint32_t off = sw128_offset((uint32_t)r, ch);
        uint4 v = *reinterpret_cast<const uint4*>(gbase + src + off);
        v.x = mul_bf16x2(v.x, w2);
        v.y = mul_bf16x2(v.y, w2);
        v.z = mul_bf16x2(v.z, w2);
        v.w = mul_bf16x2(v.w, w2);
        *reinterpret_cast<uint4*>(gbase + dst + off) = v;
      }
  #pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 gv = reinterpret_cast<const uint4*>(gbase + kOG)[tid + kThr * k];
        const uint4 hv = reinterpret_cast<const uint4*>(gbase + kOH)[tid + kThr * k];
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
  #pragma unroll
        for (int q = 0; q < 4; ++q)
          gam = fmaf(bf16lo_to_f(gw[q]), bf16lo_to_f(hw[q]), fmaf(bf16hi_to_f(gw[q]), bf16hi_to_f(hw[q]), gam));
      }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- stage 1: DX = dY Xᵀ, CB = C Bᵀ, DXᵀ = X dYᵀ, CBᵀ = B Cᵀ
    if (ok && tid == 0) {
      tc_fence_after();
      const uint64_t dX = smem_desc_sw128(sbase + kOX, 16, 1024), dDY = smem_desc_sw128(sbase + kODY, 16, 1024);
      const uint64_t dB = smem_desc_sw128(sbase + kOB, 16, 1024), dC = smem_desc_sw128(sbase + kOC, 16, 1024);
      // the transposes first (warpgroup 1, whose masks take longer), then DX, CB
      // (warpgroup 0): each warpgroup starts once its own products are in
  #pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk) mma_ss(tmem + T_DXT, dX + kk * 2u, dDY + kk * 2u, kIdSS128, kk > 0);
  #pragma unroll
      for (uint32_t kk = 0; kk < 8; ++kk)
        mma_ss(tmem + T_CBT, dB + kstep_cols(kk, kBlk), dC + kstep_cols(kk, kBlk), kIdSS128, kk > 0);
      mma_commit(bar_m1b);
  #pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk) mma_ss(tmem + T_DX, dDY + kk * 2u, dX + kk * 2u, kIdSS128, kk > 0);
  #pragma unroll
      for (uint32_t kk = 0; kk < 8; ++kk)
        mma_ss(tmem + T_CB, dC + kstep_cols(kk, kBlk), dB + kstep_cols(kk, kBlk), kIdSS128, kk > 0);
      mma_commit(bar_m1);
    }
    if (ok) ok = wait_bounded(wg == 0 ? bar_m1 : bar_m1b, ph);
    tc_fence_after();
    float rowsum = 0.f, dd = 0.f;
    if (ok && wg == 0) {
      // rows s = r of DX, CB -> M3; blocks jc > quarter lie above the diagonal
  #pragma unroll 1
      for (int jc = 0; jc < 4; ++jc) {
        const uint32_t m3a = tmem + lane_addr + T_M3 + 16u * (uint32_t)jc;
        if (jc > quarter) {
          tmem_zero16(m3a);
          continue;
        }
        uint32_t dxr[32], cbr[32], m3[16];
        tmem_ld32(tmem + lane_addr + T_DX + 32u * (uint32_t)jc, dxr);
        tmem_ld32(tmem + lane_addr + T_CB + 32u * (uint32_t)jc, cbr);
        tmem_ld_wait();
        reg_fence(dxr);
        reg_fence(cbr);
        if (jc == quarter)
          row_block<true>(dxr, cbr, cs2, dl, jc, r, cs2_r, rowsum, dd, m3);
        else
          row_block<false>(dxr, cbr, cs2, dl, jc, r, cs2_r, rowsum, dd, m3);
        tmem_st16(m3a, m3);
      }
      tmem_st_wait();
    } else if (ok) {
      // rows t = r of DXᵀ, CBᵀ -> M1ᵀ, M2ᵀ; blocks sc < quarter lie below the diagonal
      float colsum = 0.f;
  #pragma unroll 1
      for (int sc = 0; sc < 4; ++sc) {
        const uint32_t m1a = tmem + lane_addr + T_M1T + 16u * (uint32_t)sc;
        const uint32_t m2a = tmem + lane_addr + T_M2T + 16u * (uint32_t)sc;
        if (sc < quarter) {
          tmem_zero16(m1a);
          tmem_zero16(m2a);
          continue;
        }
        uint32_t dxt[32], cbt[32], m1[16], m2[16];
        tmem_ld32(tmem + lane_addr + T_DXT + 32u * (uint32_t)sc, dxt);
        tmem_ld32(tmem + lane_addr + T_CBT + 32u * (uint32_t)sc, cbt);
        tmem_ld_wait();
        reg_fence(dxt);
        reg_fence(cbt);
        if (sc == quarter)
          col_block<true>(dxt, cbt, cs2, sc, r, cs2_r, colsum, m1, m2);
        else
          col_block<false>(dxt, cbt, cs2, sc, r, cs2_r, colsum, m1, m2);
        tmem_st16(m1a, m1);
        tmem_st16(m2a, m2);
      }
      tmem_st_wait();
      vec[V_COLS + r] = dl_r * colsum;
    }
    tc_fence_before();
    ok = __syncthreads_and(ok);

    // ---- stage 2: u (M1ᵀ dY), GB = B Goutᵀ, CH = C Hinᵀ, dB (M2ᵀ C + X̃ Gout)
    if (ok && tid == 0) {
      tc_fence_after();
      const uint64_t dDYm = smem_desc_sw128(sbase + kODY, kBlk, 1024);   // dY [s][p] MN-major
      const uint64_t dB = smem_desc_sw128(sbase + kOB, 16, 1024), dC = smem_desc_sw128(sbase + kOC, 16, 1024);
      const uint64_t dG = smem_desc_sw128(sbase + kOG, 16, 1024), dH = smem_desc_sw128(sbase + kOH, 16, 1024);
      const uint64_t dCm = smem_desc_sw128(sbase + kOC, kBlk, 1024);     // C [s][n] MN-major
      const uint64_t dGm = smem_desc_sw128(sbase + kOG, kBlkS, 1024);    // Gout [p][n] MN-major
      const uint64_t dXS = smem_desc_sw128(sbase + kOXS, 16, 1024);
      // u, GB, CH first (read by warpgroup 0), then dB (warpgroup 1): each
      // warpgroup starts once its own results are in
  #pragma unroll
      for (uint32_t kk = 0; kk < 8; ++kk) {
        mma_ts(tmem + T_U, tmem + T_M1T + kk * 8u, dDYm + kk * 128u, kIdMN64, kk > 0);
        mma_ss(tmem + T_GB, dB + kstep_cols(kk, kBlk), dG + kstep_cols(kk, kBlkS), kIdSS64, kk > 0);
        mma_ss(tmem + T_CH, dC + kstep_cols(kk, kBlk), dH + kstep_cols(kk, kBlkS), kIdSS64, kk > 0);
      }
      mma_commit(bar_m2);
  #pragma unroll
      for (uint32_t kk = 0; kk < 8; ++kk)
        mma_ts(tmem + T_DB, tmem + T_M2T + kk * 8u, dCm + kk * 128u, kIdMN128, kk > 0);
  #pragma unroll
      for (uint32_t kk = 0; kk < 4; ++kk) mma_ss(tmem + T_DB, dXS + kk * 2u, dGm + kk * 128u, kIdMN128, 1);
      mma_commit(bar_m2b);
    }
    if (ok) ok = wait_bounded(wg == 0 ? bar_m2 : bar_m2b, ph);
    // warpgroup 1 stages dB in the buffer the last dC reduction read: thread 0
    // waits for that read, and warp 0 hands the all-clear to warpgroup 1 on
    // named barrier 1 (warp 0 arrives, the four warps of warpgroup 1 wait)
    if (tid == 0) tma_store_wait_read0();
    if (warp == 0)
      named_bar_arrive(1, 160);
    else if (wg == 1)
      named_bar_sync(1, 160);
    tc_fence_after();
    const int64_t tt = t0 + r;
    const bool live = tt < a.L;
    const float eg = ex2(cs2_last - cs2_r), ecs = ex2(cs2_r);
    float xu = 0.f, gbx = 0.f, a1 = 0.f;
    if (ok && wg == 0) {
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
    } else if (ok) {
      // dB row: Δ_t (M2ᵀ C + X̃ Gout), staged as four [t][32 n] boxes (128-byte
      // swizzle) that thread 0 adds into the group's accumulator in bulk
  #pragma unroll 1
      for (uint32_t nq = 0; nq < 4; ++nq) {
        uint32_t br[32];
        tmem_ld32(tmem + lane_addr + T_DB + 32u * nq, br);
        tmem_ld_wait();
        reg_fence(br);
  #pragma unroll
        for (uint32_t q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(gbase + kOStg + nq * kBlk + sw128_offset((uint32_t)r, q)) =
              make_float4(dl_r * __uint_as_float(br[4 * q]), dl_r * __uint_as_float(br[4 * q + 1]),
                          dl_r * __uint_as_float(br[4 * q + 2]), dl_r * __uint_as_float(br[4 * q + 3]));
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    ok = __syncthreads_and(ok);
    if (ok && tid == 0) {
      // rows past L are clipped by the map (its token extent is L per batch row)
  #pragma unroll
      for (uint32_t nq = 0; nq < 4; ++nq)
        tma_reduce_add_4d(&tm_db, sbase + kOStg + nq * kBlk, (int32_t)(32 * nq), g, (int32_t)t0, (int32_t)b);
      tma_store_commit();
    }

    // ---- stage 3: dC = M3 B + Ỹ Hin
    if (ok && tid == 0) {
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
    if (ok) ok = wait_bounded(bar_m3, ph);
    if (tid == 0) tma_store_wait_read0();  // the dB reduction has read the staging buffer
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (ok && tid == 0 && item + (int64_t)gridDim.x < n_items) issue_loads(item + gridDim.x);
    if (ok) {
      // columns 64 wg .. 64 wg + 63 of the dC row
  #pragma unroll 1
      for (uint32_t nq = 2 * (uint32_t)wg; nq < 2 * (uint32_t)wg + 2; ++nq) {
        uint32_t cr[32];
        tmem_ld32(tmem + lane_addr + T_DC + 32u * nq, cr);
        tmem_ld_wait();
        reg_fence(cr);
  #pragma unroll
        for (uint32_t q = 0; q < 8; ++q)
          *reinterpret_cast<float4*>(gbase + kOStg + nq * kBlk + sw128_offset((uint32_t)r, q)) =
              make_float4(__uint_as_float(cr[4 * q]), __uint_as_float(cr[4 * q + 1]), __uint_as_float(cr[4 * q + 2]),
                          __uint_as_float(cr[4 * q + 3]));
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    if (ok && tid == 0) {
  #pragma unroll
      for (uint32_t nq = 0; nq < 4; ++nq)
        tma_reduce_add_4d(&tm_dc, sbase + kOStg + nq * kBlk, (int32_t)(32 * nq), g, (int32_t)t0, (int32_t)b);
      tma_store_commit();
    }

    // dΔ, dA, dD.  Per token k (warpgroup 0, thread k):
    //   da_k = Σ_{i<k} (cols_i − rows_i) + Σ_{s≥k} e^{cs_s} C_s·(Hinᵀ dy_s)
    //        + Σ_{j<k} Δ_j e^{cs_last − cs_j} x_j·(Gout B_j) + e^{cs_last} <Gout, Hin>
    // as block scans: inclusive warp scans, then the warps' totals.
    float v1 = 0.f, v2 = 0.f, v3 = 0.f;
    if (wg == 0) {
      v1 = vec[V_COLS + r] - rowsum;
      v2 = ecs * a1;
      v3 = dl_r * eg * gbx;
    }
    float s1 = v1, s2 = v2, s3 = v3, sg = gam, sd = dd;
  #pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float u1 = __shfl_up_sync(0xffffffffu, s1, off), u2 = __shfl_up_sync(0xffffffffu, s2, off),
                  u3 = __shfl_up_sync(0xffffffffu, s3, off);
      if (lane >= off) {
        s1 += u1;
        s2 += u2;
        s3 += u3;
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
    if (wg == 0) {
      float o1 = 0.f, o2 = 0.f, o3 = 0.f, tot2 = 0.f, gsum = 0.f;
  #pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (w < warp) {
          o1 += vec[V_WT + 8 * w + 0];
          o2 += vec[V_WT + 8 * w + 1];
          o3 += vec[V_WT + 8 * w + 2];
        }
        tot2 += vec[V_WT + 8 * w + 1];
      }
  #pragma unroll
      for (int w = 0; w < kThr / 32; ++w) gsum += vec[V_WT + 8 * w + 3];
      const float da = (s1 - v1 + o1) + (tot2 - (s2 + o2) + v2) + (s3 - v3 + o3) + ex2(cs2_last) * gsum;
      if (ok && live) a.ddt[(b * a.L + tt) * a.H + h] = fmaf(a.A[h], da, xu);
      float dAp = dl_r * da;
  #pragma unroll
      for (int off = 16; off > 0; off >>= 1) dAp += __shfl_xor_sync(0xffffffffu, dAp, off);
      if (lane == 0) vec[V_WT + 8 * warp + 5] = dAp;
    }
    __syncthreads();
    if (ok && tid == 0) {
      float dAsum = 0.f, dsum = 0.f;
      for (int w = 0; w < 4; ++w) dAsum += vec[V_WT + 8 * w + 5];
      for (int w = 0; w < kThr / 32; ++w) dsum += vec[V_WT + 8 * w + 4];
      atomicAdd(a.dA + h, dAsum);
      if (a.D && a.dD) atomicAdd(a.dD + h, dsum);
    }
    __syncthreads();  // vec and TMEM free for the next item
  }
  if (!ok && tid == 0 && a.err) atomicExch(a.err, (int32_t)SSD_ERR_TIMEOUT);
  if (tid == 0) tma_store_wait_all0();  // the last reductions have read their staging and landed
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool bwd_tc_supported(const Problem& p) {
  return p.io == SSD_DTYPE_BF16 && p.P == kPt && p.N == kNt && p.B > 0 && p.L > 0;
}

cudaError_t launch_bwd_chunk_tc(const BwdProblem& q, const float* dA_cs, const float* dt_c, const void* states_bf,
                                const void* gstates_bf, float* dB_acc, float* dC_acc, cudaStream_t s) {
  const Problem& p = q.fwd;
  if (!bwd_tc_supported(p) || p.Q != kQt) return cudaErrorNotSupported;
  const int64_t srows = p.B * p.nc * p.H * kPt;  // rows of the [..][p][n] state slabs
  if (srows > INT32_MAX) return cudaErrorNotSupported;
  CUtensorMap tx, tdy, tb, tc, tg, th, tdb, tdc;
  if (!make_tma_map_bf16(&tx, p.x, p.B, p.L, p.H * kPt, kQt) ||
      !make_tma_map_bf16(&tdy, q.dy, p.B, p.L, p.H * kPt, kQt) ||
      !make_tma_map_bf16(&tb, p.Bm, p.B, p.L, p.G * kNt, kQt) ||
      !make_tma_map_bf16(&tc, p.Cm, p.B, p.L, p.G * kNt, kQt) ||
      !make_tma_map_bf16(&tg, gstates_bf, 1, srows, kNt, kPt) ||
      !make_tma_map_bf16(&th, states_bf, 1, srows, kNt, kPt) ||
      !make_tma_map_f32_bltgn(&tdb, dB_acc, p.B, p.L, p.G, kNt, kQt) ||
      !make_tma_map_f32_bltgn(&tdc, dC_acc, p.B, p.L, p.G, kNt, kQt))
    return cudaErrorInvalidValue;
  BwdTcArgs a;
  a.A = p.A;
  a.D = p.D;
  a.dA_cs = dA_cs;
  a.dt_c = dt_c;
  a.dx = q.dx;
  a.ddt = q.ddt;
  a.dB_acc = dB_acc;
  a.dC_acc = dC_acc;
  a.dA = q.dA;
  a.dD = q.dD;
  a.B = p.B;
  a.L = p.L;
  a.H = p.H;
  a.nc = p.nc;
  a.G = (int)p.G;
  a.err = p.err;
  cudaError_t e = cudaFuncSetAttribute(bwd_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int64_t n_items = p.nc * p.H * p.B;
  const unsigned grid = (unsigned)std::min<int64_t>(n_items, std::max(sms, 1));  // one persistent CTA per SM
  bwd_chunk_tc_kernel<<<grid, kThr, kSmem, s>>>(tx, tdy, tb, tc, tg, th, tdb, tdc, a);
  return cudaGetLastError();
}

}  // namespace ssd
