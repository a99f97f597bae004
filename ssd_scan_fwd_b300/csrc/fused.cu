// fused.cu -- the whole SSD forward pass in one persistent kernel for
// sm_103a: TMA loads, tcgen05 tensor-core contractions with TMEM
// accumulators, the inter-chunk state kept on chip.
//
// Method (page "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of
// SSM)"): the recurrence h_t = α_t h_{t-1} + Δ_t B_t x_t, y_t = C_tᵀ h_t (+ D x_t)
// of §2.1.2/§2.1.1, evaluated chunk by chunk in the dual form of §2.2.1
// (Y = (L ⊙ C Bᵀ) X inside a chunk, mask L_ij = ∏_{k=j+1}^{i} α_k) with the
// state carried across chunks (block decomposition of the mask figure,
// §2.2.2).  For chunk c of one (batch b, head h), with cs the in-chunk
// running sum of log2 α (Δ·A·log2 e):
//   chunk_cumsum   cs_i, w_i = 2^(cs_last − cs_i) Δ_i, 2^cs_i, 2^cs_last   (cumsum warp)
//   chunk_scan     S = C Bᵀ                                  (MMA, M=N=K=128)
//                  M_ij = S_ij 2^(cs_i − cs_j) Δ_j  (j ≤ i)  (mask warpgroup → TMEM)
//                  Y = M X                                    (MMA, A from TMEM)
//                  Y_off = C h_inᵀ                            (MMA)
//                  y_i = Y_i + 2^cs_i Y_off,i + D x_i         (epilogue warpgroup)
//   chunk_state    S_cᵀ = Bᵀ (w ⊙ X)                          (MMA, M = N_state)
//   state_passing  h_in[c+1] = 2^cs_last h_in[c] + S_c        (epilogue, fp32 in registers)
// One CTA per SM walks (b, h) sequences chunk by chunk; the state never
// leaves the SM.  Shapes: bf16 io, P = 64, N = 128, chunk Q = 128.
//
// Warp roles (384 threads):
//   warp 0      TMA producer (C, B, X tiles of a chunk; 2-stage ring)
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warp 2      chunk_cumsum of Δ·A and the per-chunk scalars
//   warp 3      TMA store of y
//   warps 4-7   mask warpgroup: X̃ = w ⊙ X and the decay mask (thread = row)
//   warps 8-11  epilogue warpgroup: state update (thread = state row n) and
//               the y epilogue (thread = token row i)
// Every wait is bounded: on timeout the CTA raises an abort flag, records
// SSD_ERR_TIMEOUT in the workspace word, drains what it issued and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128;  // chunk length (tokens)
constexpr int kP = 64;   // head dim
constexpr int kN = 128;  // state dim
constexpr int kThreads = 384;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t kBlk = kQ * 128;  // one [128 rows][128 B] swizzled block
constexpr uint32_t kOffC = 0;        // C tile: 2 blocks (state columns 0-63, 64-127)
constexpr uint32_t kOffB = 2 * kBlk; // B tile: 2 blocks
constexpr uint32_t kOffX = 4 * kBlk; // X tile: 1 block (also the y staging tile)
constexpr uint32_t kStageBytes = 5 * kBlk;
constexpr int kStages = 2;
constexpr uint32_t kOffXt = kStages * kStageBytes;  // X̃ = w ⊙ X
constexpr uint32_t kOffHb = kOffXt + kBlk;          // bf16 copy of the carried state
constexpr uint32_t kOffScal = kOffHb + kBlk;        // per-chunk scalars, 2 slots
constexpr uint32_t kScalSlot = 4 * kQ * 4 + 128;    // cs2, ej, w, ecs [kQ] + decay
constexpr uint32_t kOffBar = kOffScal + 2 * kScalSlot;

enum : uint32_t {
  B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1,  // stage ring
  B_CSF0, B_CSF1, B_CSE0, B_CSE1,            // scalar ring
  B_SFULL, B_SEMPTY,                         // S = C Bᵀ in TMEM
  B_MFULL, B_MEMPTY,                         // mask in TMEM
  B_XTFULL, B_XTEMPTY,                       // X̃ in smem
  B_HFULL,                                   // bf16 state in smem
  B_SCFULL, B_SCEMPTY,                       // chunk state in TMEM
  B_YFULL, B_YEMPTY,                         // Y, Y_off in TMEM
  B_YST0, B_YST1,                            // y staged for the TMA store
  B_DRAIN,
  kBarCount
};
constexpr uint32_t kOffMisc = kOffBar + kBarCount * 8;  // tmem base, abort flag
constexpr uint32_t kSmemUsed = kOffMisc + 16;
constexpr uint32_t kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// ---- TMEM columns (fp32 accumulators, lane = row) ----
constexpr uint32_t kTmS = 0;       // S = C Bᵀ          128 columns
constexpr uint32_t kTmY = 128;     // Y = M X            64
constexpr uint32_t kTmYoff = 192;  // Y_off = C h_inᵀ    64
constexpr uint32_t kTmSc = 256;    // S_cᵀ               64
constexpr uint32_t kTmMask = 320;  // mask, bf16 pairs   64
constexpr uint32_t kTmCols = 512;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);    // C (K-major) · Bᵀ (K-major)
constexpr uint32_t kIdescYoff = idesc_bf16_f32(128, 64, 0, 1);  // C (K-major) · h_inᵀ (MN-major)
constexpr uint32_t kIdescSc = idesc_bf16_f32(128, 64, 1, 1);    // Bᵀ (MN-major) · X̃ (MN-major)
constexpr uint32_t kIdescY = idesc_bf16_f32(128, 64, 0, 1);     // M (TMEM) · X (MN-major)

struct FusedParams {
  const float* dt;
  const float* A;
  const float* D;
  const float* init;
  float* final_state;
  int32_t B, L, H, G, nc, units;
  int32_t* err;
  uint64_t timeout_ns;
};

struct Ctl {
  volatile uint32_t* abort;
  int32_t* err;
  uint64_t timeout;
};

// Bounded wait on an mbarrier phase.  Returns false (and raises the abort
// flag) when the phase does not complete within the timeout or another role
// already aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > c.timeout) {
      *c.abort = 1u;
      if (c.err) atomicExch(c.err, (int32_t)SSD_ERR_TIMEOUT);
      return false;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    ssd_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
                     const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](uint32_t i) { return sbase + kOffBar + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + kOffMisc + 4);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    const uint32_t counts[kBarCount] = {
        1, 1, 1, 1,          // full (expect_tx by producer), empty (store warp)
        32, 32, 256, 256,    // scalars: cumsum lanes produce, both warpgroups consume
        1, 128,              // S
        128, 1,              // mask
        128, 1,              // X̃
        128,                 // h
        1, 128,              // chunk state
        1, 128,              // Y
        128, 128,            // y staged
        1};
    for (uint32_t i = 0; i < kBarCount; ++i) mbar_init(bar(i), counts[i]);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffMisc, kTmCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_y);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int heads_per_group = p.H / p.G;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t cc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const int b = u / p.H, h = u % p.H, g = h / heads_per_group;
        for (int c = 0; c < p.nc; ++c, ++cc) {
          const uint32_t s = cc & 1u, ph = (cc >> 1) & 1u;
          if (!(ok = wait_bar(bar(B_EMPTY0 + s), ph ^ 1u, ctl))) break;
          const uint32_t st = sbase + s * kStageBytes;
          mbar_arrive_expect_tx(bar(B_FULL0 + s), kStageBytes);
          tma_load_3d(st + kOffC, &tm_c, bar(B_FULL0 + s), g * kN, c * kQ, b);
          tma_load_3d(st + kOffC + kBlk, &tm_c, bar(B_FULL0 + s), g * kN + 64, c * kQ, b);
          tma_load_3d(st + kOffB, &tm_b, bar(B_FULL0 + s), g * kN, c * kQ, b);
          tma_load_3d(st + kOffB + kBlk, &tm_b, bar(B_FULL0 + s), g * kN + 64, c * kQ, b);
          tma_load_3d(st + kOffX, &tm_x, bar(B_FULL0 + s), h * kP, c * kQ, b);
        }
      }
      if (!ok) {
        // let every load already issued land before the CTA exits
        for (uint32_t k = (cc >= 2 ? cc - 2 : 0); k < cc; ++k) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(B_FULL0 + (k & 1u)), (k >> 1) & 1u) && globaltimer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t cc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        for (int c = 0; c < p.nc; ++c, ++cc) {
          const uint32_t s = cc & 1u, ph = (cc >> 1) & 1u, cp = cc & 1u;
          const uint32_t st = sbase + s * kStageBytes;
          const uint32_t sC = st + kOffC, sB = st + kOffB, sX = st + kOffX;
          if (!(ok = wait_bar(bar(B_FULL0 + s), ph, ctl))) break;
          if (!(ok = wait_bar(bar(B_SEMPTY), cp ^ 1u, ctl))) break;
          tc_fence_after();
          // S = C Bᵀ: both operands K-major over the state dimension.
          for (uint32_t kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * kBlk + (kk & 3u) * 32u;
            mma_ss(tmem + kTmS, smem_desc_sw128(sC + koff, 16, 1024), smem_desc_sw128(sB + koff, 16, 1024),
                   kIdescS, kk > 0);
          }
          mma_commit(bar(B_SFULL));
          // Y_off = C h_inᵀ: h_in stored [n][p] (MN-major B operand, K = n).
          if (!(ok = wait_bar(bar(B_YEMPTY), cp ^ 1u, ctl))) break;
          if (!(ok = wait_bar(bar(B_HFULL), cp, ctl))) break;
          tc_fence_after();
          for (uint32_t kk = 0; kk < 8; ++kk) {
            const uint32_t koff = (kk >> 2) * kBlk + (kk & 3u) * 32u;
            mma_ss(tmem + kTmYoff, smem_desc_sw128(sC + koff, 16, 1024),
                   smem_desc_sw128(sbase + kOffHb + kk * 2048u, kBlk, 1024), kIdescYoff, kk > 0);
          }
          // S_cᵀ = Bᵀ X̃: A = B tile read MN-major (M = state rows in two
          // 64-wide atoms kBlk apart), B = X̃ MN-major; K = tokens.
          if (!(ok = wait_bar(bar(B_SCEMPTY), cp ^ 1u, ctl))) break;
          if (!(ok = wait_bar(bar(B_XTFULL), cp, ctl))) break;
          tc_fence_after();
          for (uint32_t kk = 0; kk < 8; ++kk) {
            mma_ss(tmem + kTmSc, smem_desc_sw128(sB + kk * 2048u, kBlk, 1024),
                   smem_desc_sw128(sbase + kOffXt + kk * 2048u, kBlk, 1024), kIdescSc, kk > 0);
          }
          mma_commit(bar(B_SCFULL));
          mma_commit(bar(B_XTEMPTY));
          // Y = M X: A = mask from TMEM (bf16 pairs, 8 columns per K=16), B = X MN-major.
          if (!(ok = wait_bar(bar(B_MFULL), cp, ctl))) break;
          tc_fence_after();
          for (uint32_t kk = 0; kk < 8; ++kk) {
            mma_ts(tmem + kTmY, tmem + kTmMask + kk * 8u, smem_desc_sw128(sX + kk * 2048u, kBlk, 1024), kIdescY,
                   kk > 0);
          }
          mma_commit(bar(B_YFULL));
          mma_commit(bar(B_MEMPTY));
        }
      }
      // wait for every MMA issued to finish before TMEM is released
      mma_commit(bar(B_DRAIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ chunk_cumsum
    uint32_t cc = 0;
    bool ok = true;
    const float kLog2e = 1.4426950408889634f;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const int b = u / p.H, h = u % p.H;
      const float a2 = p.A[h] * kLog2e;
      for (int c = 0; c < p.nc; ++c, ++cc) {
        const uint32_t slot = cc & 1u, sph = (cc >> 1) & 1u;
        if (!(ok = wait_bar(bar(B_CSE0 + slot), sph ^ 1u, ctl))) break;
        float d[4], cs[4];
        float run = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int t = c * kQ + 4 * lane + k;
          d[k] = (t < p.L) ? p.dt[((int64_t)b * p.L + t) * p.H + h] : 0.f;
          run += d[k] * a2;
          cs[k] = run;
        }
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += up;
        }
        const float excl = incl - run;
        const float last = __shfl_sync(0xffffffffu, incl, 31);
        float* sc = reinterpret_cast<float*>(gbase + kOffScal + slot * kScalSlot);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = 4 * lane + k;
          const float c2 = excl + cs[k];
          sc[i] = c2;                                                   // cs2
          sc[kQ + i] = d[k] > 0.f ? log2f(d[k]) - c2 : -INFINITY;       // ej
          sc[2 * kQ + i] = exp2f(last - c2) * d[k];                     // w
          sc[3 * kQ + i] = exp2f(c2);                                   // ecs
        }
        if (lane == 0) sc[4 * kQ] = exp2f(last);                        // decay
        mbar_arrive(bar(B_CSF0 + slot));
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ y store
    if (lane == 0) {
      uint32_t cc = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const int b = u / p.H, h = u % p.H;
        for (int c = 0; c < p.nc; ++c, ++cc) {
          const uint32_t s = cc & 1u, ph = (cc >> 1) & 1u;
          if (!(ok = wait_bar(bar(B_YST0 + s), ph, ctl))) break;
          tma_store_3d(&tm_y, sbase + s * kStageBytes + kOffX, h * kP, c * kQ, b);
          tma_store_commit();
          tma_store_wait_read0();
          mbar_arrive(bar(B_EMPTY0 + s));
        }
      }
      tma_store_wait_all0();
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ mask warpgroup
    const uint32_t q = warp & 3;
    const uint32_t row = 32 * q + lane;
    const uint32_t lane_addr = (32u * q) << 16;
    {
      uint32_t z[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) z[k] = 0u;
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_st16(tmem + lane_addr + kTmMask + 16u * k, z);
      tmem_st_wait();
    }
    uint32_t cc = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      for (int c = 0; c < p.nc; ++c, ++cc) {
        const uint32_t s = cc & 1u, ph = (cc >> 1) & 1u, cp = cc & 1u, slot = cc & 1u;
        if (!(ok = wait_bar(bar(B_CSF0 + slot), ph, ctl))) break;
        const float* sc = reinterpret_cast<const float*>(gbase + kOffScal + slot * kScalSlot);
        const float cs2_i = sc[row];
        const float w_i = sc[2 * kQ + row];
        // X̃ = w ⊙ X (row `row` of the chunk), same swizzled layout as X.
        if (!(ok = wait_bar(bar(B_FULL0 + s), ph, ctl))) break;
        if (!(ok = wait_bar(bar(B_XTEMPTY), cp ^ 1u, ctl))) break;
        const uint32_t sX = sbase + s * kStageBytes + kOffX;
#pragma unroll
        for (uint32_t ch = 0; ch < 8; ++ch) {
          const uint32_t off = sw128_offset(row, ch);
          uint32_t v[4];
          ld_shared_v4(sX + off, v[0], v[1], v[2], v[3]);
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] = pack_bf16x2(bf16lo_to_f(v[k]) * w_i, bf16hi_to_f(v[k]) * w_i);
          st_shared_v4(sbase + kOffXt + off, v[0], v[1], v[2], v[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_XTFULL));
        // Decay mask from S = C Bᵀ, column slabs of 32 on or below the diagonal.
        if (!(ok = wait_bar(bar(B_SFULL), cp, ctl))) break;
        if (!(ok = wait_bar(bar(B_MEMPTY), cp ^ 1u, ctl))) break;
        tc_fence_after();
        for (uint32_t k = 0; k <= q; ++k) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_addr + kTmS + 32u * k, r);
          tmem_ld_wait();
          uint32_t m[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const int j = 32 * k + e;
            float v0 = __uint_as_float(r[e]) * exp2f(cs2_i + sc[kQ + j]);
            float v1 = __uint_as_float(r[e + 1]) * exp2f(cs2_i + sc[kQ + j + 1]);
            if (j > (int)row) v0 = 0.f;
            if (j + 1 > (int)row) v1 = 0.f;
            m[e >> 1] = pack_bf16x2(v0, v1);
          }
          tmem_st16(tmem + lane_addr + kTmMask + 16u * k, m);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(B_SEMPTY));
        mbar_arrive(bar(B_MFULL));
        mbar_arrive(bar(B_CSE0 + slot));
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue warpgroup
    const uint32_t q = warp & 3;
    const uint32_t row = 32 * q + lane;  // state row n for the update, token row i for y
    const uint32_t lane_addr = (32u * q) << 16;
    uint32_t cc = 0;
    bool ok = true;
    float hs[kP];
    for (int u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
      const int b = u / p.H, h = u % p.H;
      const float Dh = p.D ? p.D[h] : 0.f;
      const int64_t st_off = ((int64_t)b * p.H + h) * kP * kN;
      // state entering the sequence, row n = `row` of hᵀ
#pragma unroll
      for (int pp = 0; pp < kP; ++pp) hs[pp] = p.init ? p.init[st_off + (int64_t)pp * kN + row] : 0.f;
      auto write_hb = [&]() {
#pragma unroll
        for (uint32_t ch = 0; ch < 8; ++ch) {
          st_shared_v4(sbase + kOffHb + sw128_offset(row, ch), pack_bf16x2(hs[8 * ch + 0], hs[8 * ch + 1]),
                       pack_bf16x2(hs[8 * ch + 2], hs[8 * ch + 3]), pack_bf16x2(hs[8 * ch + 4], hs[8 * ch + 5]),
                       pack_bf16x2(hs[8 * ch + 6], hs[8 * ch + 7]));
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_HFULL));
      };
      write_hb();
      for (int c = 0; c < p.nc; ++c, ++cc) {
        const uint32_t s = cc & 1u, ph = (cc >> 1) & 1u, cp = cc & 1u, slot = cc & 1u;
        if (!(ok = wait_bar(bar(B_CSF0 + slot), ph, ctl))) break;
        const float* sc = reinterpret_cast<const float*>(gbase + kOffScal + slot * kScalSlot);
        const float decay = sc[4 * kQ];
        const float ecs_i = sc[3 * kQ + row];
        // state_passing: h_in[c+1] = decay h_in[c] + S_c
        if (!(ok = wait_bar(bar(B_SCFULL), cp, ctl))) break;
        tc_fence_after();
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tmem + lane_addr + kTmSc, r0);
          tmem_ld32(tmem + lane_addr + kTmSc + 32u, r1);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(bar(B_SCEMPTY));
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            hs[k] = fmaf(decay, hs[k], __uint_as_float(r0[k]));
            hs[32 + k] = fmaf(decay, hs[32 + k], __uint_as_float(r1[k]));
          }
        }
        if (c + 1 < p.nc) write_hb();
        // y epilogue, in two halves of 32 columns to bound register use
        if (!(ok = wait_bar(bar(B_YFULL), cp, ctl))) break;
        if (!(ok = wait_bar(bar(B_FULL0 + s), ph, ctl))) break;
        tc_fence_after();
        const uint32_t sX = sbase + s * kStageBytes + kOffX;
#pragma unroll
        for (uint32_t half = 0; half < 2; ++half) {
          uint32_t ya[32], oa[32];
          tmem_ld32(tmem + lane_addr + kTmY + 32u * half, ya);
          tmem_ld32(tmem + lane_addr + kTmYoff + 32u * half, oa);
          tmem_ld_wait();
          if (half == 1) {
            tc_fence_before();
            mbar_arrive(bar(B_YEMPTY));
          }
#pragma unroll
          for (uint32_t cq = 0; cq < 4; ++cq) {
            const uint32_t ch = 4 * half + cq;
            const uint32_t off = sw128_offset(row, ch);
            uint32_t v[4];
            ld_shared_v4(sX + off, v[0], v[1], v[2], v[3]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = 8 * cq + 2 * k;  // column within the half
              const float r0 = __uint_as_float(ya[e]) + ecs_i * __uint_as_float(oa[e]) + Dh * bf16lo_to_f(v[k]);
              const float r1 =
                  __uint_as_float(ya[e + 1]) + ecs_i * __uint_as_float(oa[e + 1]) + Dh * bf16hi_to_f(v[k]);
              v[k] = pack_bf16x2(r0, r1);
            }
            st_shared_v4(sX + off, v[0], v[1], v[2], v[3]);
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_YST0 + s));
        mbar_arrive(bar(B_CSE0 + slot));
      }
      if (ok && p.final_state) {
#pragma unroll
        for (int pp = 0; pp < kP; ++pp) p.final_state[st_off + (int64_t)pp * kN + row] = hs[pp];
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D bf16 tensor map over [B][L][W] (W = row width in elements), box
// [1][128][64] with the 128-byte swizzle; rows past L read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t W) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)(W * 2), (cuuint64_t)(L * W * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)kQ, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- static scratch
// Scratch for ssd_fwd_noalloc: a fixed device array in the library image, so
// callers that must not allocate device memory still have somewhere for the
// fused kernel's workspace word.  Every GPU that loads the library holds it
// until the process exits.
constexpr size_t kStaticScratchBytes = size_t(1) << 20;  // 1 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

}  // namespace

size_t static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of g_static_scratch on the current device.  Resolved once
// per device (with that device current) by cudaGetSymbolAddress; in host code
// the array's name is only a host-side stand-in, never a device address.
cudaError_t static_scratch_ptr(void** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

bool fused_supported(const Problem& p) {
  return p.io == SSD_DTYPE_BF16 && p.P == kP && p.N == kN && (p.Q_req == 0 || p.Q_req == kQ) &&
         p.B * p.H < (int64_t(1) << 31) && p.L < (int64_t(1) << 31) && encode_fn() != nullptr;
}

size_t fused_workspace_bytes(const Problem&) { return 256; }

cudaError_t launch_fused(const Problem& p, void* workspace, cudaStream_t s) {
  CUtensorMap tx, tb, tc, ty;
  if (!make_map(&tx, p.x, p.B, p.L, p.H * kP) || !make_map(&tb, p.Bm, p.B, p.L, p.G * kN) ||
      !make_map(&tc, p.Cm, p.B, p.L, p.G * kN) || !make_map(&ty, p.y, p.B, p.L, p.H * kP))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(ssd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemAlloc)) != cudaSuccess)
    return e;
  if ((e = cudaMemsetAsync(workspace, 0, 256, s)) != cudaSuccess) return e;
  FusedParams fp;
  fp.dt = p.dt;
  fp.A = p.A;
  fp.D = p.D;
  fp.init = p.init;
  fp.final_state = p.final_state;
  fp.B = (int32_t)p.B;
  fp.L = (int32_t)p.L;
  fp.H = (int32_t)p.H;
  fp.G = (int32_t)p.G;
  fp.nc = (int32_t)((p.L + kQ - 1) / kQ);
  fp.units = (int32_t)(p.B * p.H);
  fp.err = static_cast<int32_t*>(workspace);
  fp.timeout_ns = 2000000000ull;
  const int grid = (int)std::min<int64_t>(fp.units, sms);
  ssd_fused_kernel<<<grid, kThreads, kSmemAlloc, s>>>(tx, tb, tc, ty, fp);
  return cudaGetLastError();
}

}  // namespace ssd
