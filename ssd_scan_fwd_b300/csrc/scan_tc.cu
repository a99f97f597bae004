// scan_tc.cu -- the chunk outputs (step 4 of the chunked form) on the tensor
// cores: bf16 io, headdim 64, dstate 16, 64, 128 or 256, chunk 128, real or
// complex decay.
//
// For chunk c of head h with token rows i, j = 0..127 ("Mamba-3 深度剖析 -
// 02. SSM 基础回顾与演进", §2.2.1: the masked quadratic form inside a chunk
// plus the read-out of the state entering it):
//   S = C Bᵀ,   M[i][j] = S[i][j] e^{cs_i − cs_j} Δ_j (j ≤ i)
//   y_i = (M X)_i + e^{cs_i} C_i·h_in + D x_i
// and, with the complex decay (rotation angles φ = in-chunk sums of θ),
//   M[i][j] gains cos(φ_i − φ_j) = cos φ_i cos φ_j + sin φ_i sin φ_j and the
//   read-out is e^{cs_i}(cos φ_i C_i·Re h_in − sin φ_i C_i·Im h_in).
// An optional gate multiplies y by silu(z).
//
// One CTA of 256 threads per (chunk, head, batch row), two per SM up to
// dstate 128 (99 KB of shared memory at 128, 256 TMEM columns), one at 256.
// TMA brings C, B, X and the bf16 copy of Re h_in written by the state
// recurrence.  One thread issues S = C Bᵀ
// (TMEM columns 0-127) and R = C Re h_inᵀ (128-191); with the complex decay,
// once S is done, Im h_in is loaded over the B tile and I = C Im h_inᵀ goes
// to 192-255.  Token row i is TMEM lane i; the two warpgroups split the four
// 32-column blocks of the row, turn them into M (bf16, written over S's first
// 64 columns; blocks above the diagonal are stored as zeros unread), and
// Y = M X (A from TMEM) goes to columns 64-127.  The epilogue reads Y, R (and
// I) for its 32 columns of y and stores them with 16-byte accesses.
// Exponentials are ex2 of the running sums prescaled by log2 e.  Waits are
// bounded (2 s).

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <cstdlib>

#include "internal.h"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kQs = 128, kPs = 64, kThr = 256;
constexpr uint32_t kBlk = kQs * 128;     // [128 rows][64 columns] swizzled block
constexpr uint32_t kBlkS = kPs * 128;    // [64 rows][64 columns]
enum : int { V_CS2 = 0, V_DL = 128, V_CPH = 256, V_SPH = 384, V_COUNT = 512 };

// Shared memory for dstate NS (NS / 64 column blocks per tile; one block,
// zero past column NS, at NS = 16).
template <int NS>
struct ScanTcSmem {
  static constexpr uint32_t kNB = NS < 64 ? 1 : NS / 64;
  static constexpr uint32_t kOC = 0;                   // C [i][n]
  static constexpr uint32_t kOB = kNB * kBlk;          // B [j][n]; later Im h_in [p][n]
  static constexpr uint32_t kOX = 2 * kNB * kBlk;      // X [j][p]
  static constexpr uint32_t kOH = kOX + kBlk;          // Re h_in (bf16) [p][n]
  static constexpr uint32_t kOV = kOH + kNB * kBlkS;
  static constexpr uint32_t kOBar = kOV + V_COUNT * 4;
  static constexpr uint32_t kOMisc = kOBar + 4 * 8;
  static constexpr uint32_t kSmem = kOMisc + 16 + 1024;
  static constexpr uint32_t kLoadBytes = (2 * kNB + 1) * kBlk + kNB * kBlkS;
  static constexpr int kMinBlocks = NS <= 128 ? 2 : 1;
  static_assert(kSmem * kMinBlocks <= 228 * 1024 - kMinBlocks * 1024, "CTAs per SM");
};

constexpr uint32_t T_S = 0, T_M = 0, T_Y = 64, T_R = 128, T_I = 192;
constexpr uint32_t kIdS = idesc_bf16_f32(128, 128, 0, 0);   // C (K-major) · Bᵀ (K-major)
constexpr uint32_t kIdR = idesc_bf16_f32(128, 64, 0, 0);    // C (K-major) · h_inᵀ (K-major)
constexpr uint32_t kIdY = idesc_bf16_f32(128, 64, 0, 1);    // M (TMEM) · X (MN-major)

struct ScanTcArgs {
  const float* D;
  const float* dA_cs;
  const float* dt_c;
  const float* phi;
  const __nv_bfloat16* z;
  __nv_bfloat16* y;
  int64_t L, H, nc;
  int G;
  int32_t* err;  // SSD_ERR_TIMEOUT is written here when a bounded wait gives up (may be null)
};

// M for the 32 columns j = 32 jc .. of row i.  kDiag: the block holding the
// diagonal (j ≤ i kept).
template <bool kRot, bool kDiag>
__device__ __forceinline__ void mask_block(const uint32_t (&sr)[32], const float* vec, int jc, int i, float cs2_i,
                                           float cph_i, float sph_i, uint32_t (&m)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float v[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int j = 32 * jc + e + q;
      float w = __uint_as_float(sr[e + q]) * ex2(cs2_i - vec[V_CS2 + j]) * vec[V_DL + j];
      if (kRot) w *= fmaf(cph_i, vec[V_CPH + j], sph_i * vec[V_SPH + j]);
      if (kDiag && j > i) w = 0.f;
      v[q] = w;
    }
    m[e >> 1] = pack_bf16x2(v[0], v[1]);
  }
}

template <bool kRot>
__device__ __forceinline__ void mask_one(uint32_t tmem, uint32_t lane_addr, int jc, int quarter, const float* vec,
                                         int r, float cs2_r, float cph, float sph, const uint32_t (&sr)[32]) {
  uint32_t m[16];
  if (jc == quarter)
    mask_block<kRot, true>(sr, vec, jc, r, cs2_r, cph, sph, m);
  else
    mask_block<kRot, false>(sr, vec, jc, r, cs2_r, cph, sph, m);
  tmem_st16(tmem + lane_addr + T_M + 16u * (uint32_t)jc, m);
}

template <bool kRot, int NS>
__global__ void __launch_bounds__(kThr, ScanTcSmem<NS>::kMinBlocks)
    chunk_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_hr,
                         const __grid_constant__ CUtensorMap tm_hi, const ScanTcArgs a) {
  using Sm = ScanTcSmem<NS>;
  constexpr uint32_t kNB = Sm::kNB, kOC = Sm::kOC, kOB = Sm::kOB, kOX = Sm::kOX, kOH = Sm::kOH;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  float* vec = reinterpret_cast<float*>(gbase + Sm::kOV);
  const uint32_t bar_load = sbase + Sm::kOBar, bar_s = bar_load + 8, bar_hi = bar_load + 16, bar_y = bar_load + 24;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + Sm::kOMisc);

  const int64_t c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = (int)(h / (a.H / a.G));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = warp >> 2, quarter = warp & 3;
  const int r = 32 * quarter + lane;
  const uint32_t lane_addr = (32u * (uint32_t)quarter) << 16;
  const int64_t t0 = c * kQs;
  const int32_t srow = (int32_t)(((b * a.nc + c) * a.H + h) * kPs);  // row of the [p][n] state slabs

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_hi, 1);
    mbar_init(bar_y, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + Sm::kOMisc, 256);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, Sm::kLoadBytes);
#pragma unroll
    for (uint32_t k = 0; k < kNB; ++k) {
      if (NS < 64) {  // [B][L][G][N] maps: coordinates (0, g, t, b)
        tma_load_4d(sbase + kOC, &tm_c, bar_load, 0, g, (int32_t)t0, (int32_t)b);
        tma_load_4d(sbase + kOB, &tm_b, bar_load, 0, g, (int32_t)t0, (int32_t)b);
      } else {
        tma_load_3d(sbase + kOC + k * kBlk, &tm_c, bar_load, g * NS + 64 * (int)k, (int32_t)t0, (int32_t)b);
        tma_load_3d(sbase + kOB + k * kBlk, &tm_b, bar_load, g * NS + 64 * (int)k, (int32_t)t0, (int32_t)b);
      }
      tma_load_3d(sbase + kOH + k * kBlkS, &tm_hr, bar_load, 64 * (int)k, srow, 0);
    }
    tma_load_3d(sbase + kOX, &tm_x, bar_load, (int32_t)(h * kPs), (int32_t)t0, (int32_t)b);
  }
  {
    const int64_t vrow = ((b * a.H + h) * a.nc + c) * kQs;
    if (wg == 0) {
      vec[V_CS2 + r] = a.dA_cs[vrow + r] * kLog2e;
      vec[V_DL + r] = a.dt_c[vrow + r];
    } else if (kRot) {
      float sv, cv;
      sincosf(a.phi[vrow + r], &sv, &cv);
      vec[V_CPH + r] = cv;
      vec[V_SPH + r] = sv;
    }
  }
  bool ok = __syncthreads_and(wait_bounded(bar_load, 0));
  // S = C Bᵀ, R = C Re h_inᵀ
  if (ok && tid == 0) {
    tc_fence_after();
    const uint64_t dC = smem_desc_sw128(sbase + kOC, 16, 1024), dB = smem_desc_sw128(sbase + kOB, 16, 1024);
    const uint64_t dH = smem_desc_sw128(sbase + kOH, 16, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < NS / 16; ++kk)
      mma_ss(tmem + T_S, dC + kstep_cols(kk, kBlk), dB + kstep_cols(kk, kBlk), kIdS, kk > 0);
#pragma unroll
    for (uint32_t kk = 0; kk < NS / 16; ++kk)
      mma_ss(tmem + T_R, dC + kstep_cols(kk, kBlk), dH + kstep_cols(kk, kBlkS), kIdR, kk > 0);
    mma_commit(bar_s);
  }
  if (ok) ok = wait_bounded(bar_s, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (kRot && ok && tid == 0) {
    // the B tile is free once S is done: Im h_in goes over it
    mbar_arrive_expect_tx(bar_hi, kNB * kBlkS);
#pragma unroll
    for (uint32_t k = 0; k < kNB; ++k) tma_load_3d(sbase + kOB + k * kBlkS, &tm_hi, bar_hi, 64 * (int)k, srow, 0);
  }
  const float cs2_r = vec[V_CS2 + r];
  const float cph = kRot ? vec[V_CPH + r] : 1.f, sph = kRot ? vec[V_SPH + r] : 0.f;
  // mask: warpgroup 0 takes column blocks 0 and 1, warpgroup 1 blocks 2 and 3.
  // M is written over S's columns 0-63, which hold blocks 0 and 1 of S, so
  // warpgroup 0 loads both its blocks before anyone writes.
  uint32_t s0[32], s1[32];
  if (ok && wg == 0) {
    if (quarter >= 0) tmem_ld32(tmem + lane_addr + T_S, s0);
    if (quarter >= 1) tmem_ld32(tmem + lane_addr + T_S + 32u, s1);
    tmem_ld_wait();
    reg_fence(s0);
    reg_fence(s1);
  }
  __syncthreads();
  if (ok && wg == 0) {
    mask_one<kRot>(tmem, lane_addr, 0, quarter, vec, r, cs2_r, cph, sph, s0);
    if (quarter >= 1)
      mask_one<kRot>(tmem, lane_addr, 1, quarter, vec, r, cs2_r, cph, sph, s1);
    else
      tmem_zero16(tmem + lane_addr + T_M + 16u);
    tmem_st_wait();
  } else if (ok) {
#pragma unroll 1
    for (int jc = 2; jc < 4; ++jc) {
      if (jc > quarter) {
        tmem_zero16(tmem + lane_addr + T_M + 16u * (uint32_t)jc);
        continue;
      }
      tmem_ld32(tmem + lane_addr + T_S + 32u * (uint32_t)jc, s0);
      tmem_ld_wait();
      reg_fence(s0);
      mask_one<kRot>(tmem, lane_addr, jc, quarter, vec, r, cs2_r, cph, sph, s0);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  // Y = M X (columns 64-127, over S's blocks 2 and 3, read above); I = C Im h_inᵀ
  if (ok && tid == 0) {
    tc_fence_after();
    const uint64_t dXm = smem_desc_sw128(sbase + kOX, kBlk, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < 8; ++kk) mma_ts(tmem + T_Y, tmem + T_M + kk * 8u, dXm + kk * 128u, kIdY, kk > 0);
    if (kRot) {
      if (wait_bounded(bar_hi, 0)) {
        tc_fence_after();
        const uint64_t dC = smem_desc_sw128(sbase + kOC, 16, 1024), dI = smem_desc_sw128(sbase + kOB, 16, 1024);
#pragma unroll
        for (uint32_t kk = 0; kk < NS / 16; ++kk)
          mma_ss(tmem + T_I, dC + kstep_cols(kk, kBlk), dI + kstep_cols(kk, kBlkS), kIdR, kk > 0);
      }
    }
    mma_commit(bar_y);
  }
  if (ok) ok = wait_bounded(bar_y, 0);
  if (kRot && ok) ok = mbar_test_wait(bar_hi, 0);  // I issued (not skipped on a timeout)
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    const int64_t tt = t0 + r;
    const bool live = tt < a.L;
    const float ecs = ex2(cs2_r);
    const float kr = ecs * cph, ki = -ecs * sph;
    const float Dh = a.D ? a.D[h] : 0.f;
#pragma unroll 1
    for (uint32_t k = 0; k < 2; ++k) {
      const uint32_t col = 32u * (uint32_t)wg + 16u * k;  // p of the first of 16 columns
      uint32_t yr[16], rr[16], ir[16];
      tmem_ld16(tmem + lane_addr + T_Y + col, yr);
      tmem_ld16(tmem + lane_addr + T_R + col, rr);
      if (kRot) tmem_ld16(tmem + lane_addr + T_I + col, ir);
      tmem_ld_wait();
      reg_fence16(yr);
      reg_fence16(rr);
      if (kRot) reg_fence16(ir);
      if (!live) continue;
      const int64_t o = ((b * a.L + tt) * a.H + h) * kPs + col;
      uint4 zv[2];
      if (a.z) {
        zv[0] = reinterpret_cast<const uint4*>(a.z + o)[0];
        zv[1] = reinterpret_cast<const uint4*>(a.z + o)[1];
      }
      uint32_t out[8];
#pragma unroll
      for (uint32_t ch = 0; ch < 2; ++ch) {
        const uint4 xv = *reinterpret_cast<const uint4*>(gbase + kOX + sw128_offset((uint32_t)r, col / 8 + ch));
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t zw[4] = {zv[ch].x, zv[ch].y, zv[ch].z, zv[ch].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = 8 * (int)ch + 2 * q;
          float v0 = fmaf(kr, __uint_as_float(rr[e]), fmaf(Dh, bf16lo_to_f(xw[q]), __uint_as_float(yr[e])));
          float v1 = fmaf(kr, __uint_as_float(rr[e + 1]), fmaf(Dh, bf16hi_to_f(xw[q]), __uint_as_float(yr[e + 1])));
          if (kRot) {
            v0 = fmaf(ki, __uint_as_float(ir[e]), v0);
            v1 = fmaf(ki, __uint_as_float(ir[e + 1]), v1);
          }
          if (a.z) {  // gate: y · silu(z)
            const float z0 = bf16lo_to_f(zw[q]), z1 = bf16hi_to_f(zw[q]);
            v0 *= z0 / (1.f + expf(-z0));
            v1 *= z1 / (1.f + expf(-z1));
          }
          out[4 * ch + q] = pack_bf16x2(v0, v1);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(a.y + o);
      dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
      dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
  }
  if (!ok && tid == 0 && a.err) atomicExch(a.err, (int32_t)SSD_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace

bool scan_tc_supported(const Problem& p) {
  const bool n_ok = p.N == 16 || p.N == 64 || p.N == 128 || p.N == 256;
  if (!(p.io == SSD_DTYPE_BF16 && p.P == kPs && n_ok && p.Q == kQs && p.B > 0 && p.L > 0)) return false;
  const char* env = getenv("SSD_CHUNK_SCAN_CUDA_CORES");
  return !(env && atoi(env) == 1);
}

cudaError_t launch_chunk_scan_tc(const Problem& p, const float* dA_cs, const float* dt_c, const float* phi,
                                 const void* re_bf, const void* im_bf, cudaStream_t s) {
  if (!scan_tc_supported(p)) return cudaErrorNotSupported;
  const bool rot = phi != nullptr;
  if (rot && !im_bf) return cudaErrorInvalidValue;
  const int64_t srows = p.B * p.nc * p.H * kPs;
  if (srows > INT32_MAX) return cudaErrorNotSupported;
  CUtensorMap tc, tb, tx, thr, thi;
  const bool narrow = p.N < 64;
  auto map_bc = [&](CUtensorMap* m, const void* base) {
    return narrow ? make_tma_map_bf16_narrow(m, base, p.B, p.L, p.G, p.N, kQs)
                  : make_tma_map_bf16(m, base, p.B, p.L, p.G * p.N, kQs);
  };
  if (!map_bc(&tc, p.Cm) || !map_bc(&tb, p.Bm) ||
      !make_tma_map_bf16(&tx, p.x, p.B, p.L, p.H * kPs, kQs) ||
      !make_tma_map_bf16(&thr, re_bf, 1, srows, p.N, kPs) ||
      !make_tma_map_bf16(&thi, rot ? im_bf : re_bf, 1, srows, p.N, kPs))
    return cudaErrorInvalidValue;
  ScanTcArgs a;
  a.D = p.D;
  a.dA_cs = dA_cs;
  a.dt_c = dt_c;
  a.phi = phi;
  a.z = static_cast<const __nv_bfloat16*>(p.z);
  a.y = static_cast<__nv_bfloat16*>(p.y);
  a.L = p.L;
  a.H = p.H;
  a.nc = p.nc;
  a.G = (int)p.G;
  a.err = p.err;
  dim3 grid((unsigned)p.nc, (unsigned)p.H, (unsigned)p.B);
  auto run = [&](auto kernel, uint32_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThr, smem, s>>>(tc, tb, tx, thr, thi, a);
    return cudaGetLastError();
  };
  switch (p.N) {
    case 16: return rot ? run(chunk_scan_tc_kernel<true, 16>, ScanTcSmem<16>::kSmem)
                        : run(chunk_scan_tc_kernel<false, 16>, ScanTcSmem<16>::kSmem);
    case 64: return rot ? run(chunk_scan_tc_kernel<true, 64>, ScanTcSmem<64>::kSmem)
                        : run(chunk_scan_tc_kernel<false, 64>, ScanTcSmem<64>::kSmem);
    case 128: return rot ? run(chunk_scan_tc_kernel<true, 128>, ScanTcSmem<128>::kSmem)
                         : run(chunk_scan_tc_kernel<false, 128>, ScanTcSmem<128>::kSmem);
    case 256: return rot ? run(chunk_scan_tc_kernel<true, 256>, ScanTcSmem<256>::kSmem)
                         : run(chunk_scan_tc_kernel<false, 256>, ScanTcSmem<256>::kSmem);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace ssd
