// state_tc.cu -- the chunk states of the chunked path on the tensor cores
// (bf16 io, headdim 64, dstate 16, 64, 128 or 256, chunk 64 or 128).
//
// For chunk c of head h (page "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进",
// §2.2.1's mask restricted to "from token i to the chunk end"):
//     S_c[p][n] = Σ_i w_i x_i[p] B_i[n]
// with the weight w_i by mode: exp(cs_{Q-1} − cs_i) Δ_i (the chunk states of
// the forward pass), exp(cs_i) with x := dy, B := C (the backward pass's
// adjoint chunk states), or exp(cs_{Q-1} − cs_i) cos / sin(φ_{Q-1} − φ_i) Δ_i
// (real / imaginary chunk states of the complex decay).
//
// Dstate 128: one CTA per (chunk, head pair of a group, batch row): TMA
// brings the B tile [Q tokens][128 state columns] and the two heads' X tiles
// [Q][64] (128-byte swizzle); 128 threads scale the X rows by w in place (X̃); one thread issues
// S_cᵀ = Bᵀ · [X̃_0 | X̃_1] as Q/16 128×128×16 tcgen05 MMAs (B read MN-major
// with M = state rows, X̃ MN-major with N = both heads' 64 columns), fp32 in
// TMEM; thread n then reads state row n of both heads and stores it, each
// store coalesced over n.  Waits are bounded (2 s): a CTA that gives up
// writes nothing.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <mutex>
#include <type_traits>

#include "internal.h"
#include "sm100.cuh"
#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kPs = 64;     // head dim: N of the MMA is two heads' 64
constexpr int kNs = 128;    // state dim: M of the MMA
constexpr int kThr = 128;   // thread = state row n = TMEM lane

// Shared memory for chunk length Q (the K of the MMA).  At most four CTAs
// per SM (50 KB at Q = 64; 72 KB at Q = 128 allows three), so that their
// 128-column TMEM allocations always fit the 512 columns.
template <int Q>
struct TcSmem {
  static constexpr uint32_t kBlk = Q * 128;          // one [Q rows][128 B] swizzled block
  static constexpr uint32_t kOffB = 0;               // B tile: state columns 0-63, 64-127
  static constexpr uint32_t kOffX = 2 * kBlk;        // X tiles of head 0, head 1
  static constexpr uint32_t kOffW = 4 * kBlk;        // weights [2][Q] fp32
  static constexpr uint32_t kOffBar = kOffW + 2 * Q * 4;
  static constexpr uint32_t kOffMisc = kOffBar + 2 * 8;
  static constexpr uint32_t kBytes = Q == 64 ? 50 * 1024 : 72 * 1024;
  static_assert(kOffMisc + 16 + 1024 <= kBytes, "shared memory layout");
};
constexpr uint32_t kIdescTc = idesc_bf16_f32(128, 128, 1, 1);  // Bᵀ (MN-major) · X̃ (MN-major)

template <int Q, int kMode>
__global__ void __launch_bounds__(kThr) chunk_state_tc_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                             const __grid_constant__ CUtensorMap tm_b,
                                                             const float* __restrict__ dA_cs,
                                                             const float* __restrict__ dt_c,
                                                             const float* __restrict__ phi, int64_t L, int64_t H,
                                                             int G, int64_t nc, int pairs_per_group,
                                                             float* __restrict__ states, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  using S = TcSmem<Q>;
  constexpr uint32_t kBlkS = S::kBlk, kOffB = S::kOffB, kOffX = S::kOffX, kOffMisc = S::kOffMisc;
  const uint32_t bar_load = sbase + S::kOffBar, bar_mma = sbase + S::kOffBar + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + kOffMisc);
  float* wsm = reinterpret_cast<float*>(gbase + S::kOffW);

  const int64_t c = blockIdx.x, b = blockIdx.z;
  const int g = (int)blockIdx.y / pairs_per_group, pr = (int)blockIdx.y % pairs_per_group;
  const int hpg = (int)(H / G);
  const int h0 = g * hpg + 2 * pr;
  const bool valid1 = 2 * pr + 1 < hpg;
  const int h1 = valid1 ? h0 + 1 : h0;
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + kOffMisc, 128);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, 4 * kBlkS);
    tma_load_3d(sbase + kOffB, &tm_b, bar_load, g * kNs, (int32_t)(c * Q), (int32_t)b);
    tma_load_3d(sbase + kOffB + kBlkS, &tm_b, bar_load, g * kNs + 64, (int32_t)(c * Q), (int32_t)b);
    tma_load_3d(sbase + kOffX, &tm_x, bar_load, h0 * kPs, (int32_t)(c * Q), (int32_t)b);
    tma_load_3d(sbase + kOffX + kBlkS, &tm_x, bar_load, h1 * kPs, (int32_t)(c * Q), (int32_t)b);
  }
  // weights of both heads' Q tokens
  for (int e = tid; e < 2 * Q; e += kThr) {
    const int hh = e / Q, i = e % Q;
    const int64_t row = ((b * H + (hh ? h1 : h0)) * nc + c) * Q;
    const float cs_i = dA_cs[row + i];
    float w;
    if (kMode == 1) {
      w = expf(cs_i);
    } else {
      w = expf(dA_cs[row + Q - 1] - cs_i) * dt_c[row + i];
      if (kMode == 2) w *= cosf(phi[row + Q - 1] - phi[row + i]);
      if (kMode == 3) w *= sinf(phi[row + Q - 1] - phi[row + i]);
    }
    wsm[e] = w;
  }
  bool ok = __syncthreads_and(wait_bounded(bar_load, 0));
  if (ok) {
    // X̃ = w ⊙ X in place: one (head, token row) per thread and pass
    for (int e = tid; e < 2 * Q; e += kThr) {
      const int hh = e / Q, r = e % Q;
      uint4* xt = reinterpret_cast<uint4*>(gbase + kOffX + hh * kBlkS);
      const float wv = wsm[e];
      const uint32_t wx = pack_bf16x2(wv, wv);
#pragma unroll
      for (uint32_t ch = 0; ch < 8; ++ch) {
        uint4 v = xt[sw128_offset((uint32_t)r, ch) >> 4];
        v.x = mul_bf16x2(v.x, wx);
        v.y = mul_bf16x2(v.y, wx);
        v.z = mul_bf16x2(v.z, wx);
        v.w = mul_bf16x2(v.w, wx);
        xt[sw128_offset((uint32_t)r, ch) >> 4] = v;
      }
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (ok && tid == 0) {
    tc_fence_after();
    const uint64_t da = smem_desc_sw128(sbase + kOffB, kBlkS, 1024);
    const uint64_t db = smem_desc_sw128(sbase + kOffX, kBlkS, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < Q / 16; ++kk) mma_ss(tmem, da + kk * 128u, db + kk * 128u, kIdescTc, kk > 0);
    mma_commit(bar_mma);
  }
  if (ok) ok = wait_bounded(bar_mma, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    // thread n: state row n of both heads, 32 columns per load
    const uint32_t lane_addr = (32u * (uint32_t)warp) << 16;
    const int n = tid;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_addr + 32u * q, r);
      tmem_ld_wait();
      reg_fence(r);
      const int hh = q >> 1;
      if (hh == 1 && !valid1) continue;
      float* dst = states + ((b * nc + c) * H + (hh ? h1 : h0)) * (int64_t)kPs * kNs;
      const int p0 = 32 * (q & 1);
#pragma unroll
      for (int e = 0; e < 32; ++e) dst[(int64_t)(p0 + e) * kNs + n] = __uint_as_float(r[e]);
    }
  }
  if (!ok && tid == 0 && err) atomicExch(err, (int32_t)SSD_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// Other state sizes (NS = 16, 64 or 256): S_c = [X̃_0 | X̃_1]ᵀ · B, the two
// heads' X̃ read MN-major as A with M = both heads' 64 rows p, the B tile
// MN-major with N = NS state columns (at NS = 16 one 64-column block whose
// columns past 16 the tensor map fills with zeros).  Thread m reads row m
// (head m / 64, p = m mod 64) of the NS fp32 columns and stores it as
// contiguous 64- or 128-byte pieces.
template <int Q, int NS>
struct TcSmem2 {
  static constexpr uint32_t kBlk = Q * 128;             // [Q rows][64 columns] swizzled block
  static constexpr uint32_t kNB = NS < 64 ? 1 : NS / 64;
  static constexpr uint32_t kOffB = 0;                  // B tile: kNB blocks
  static constexpr uint32_t kOffX = kNB * kBlk;         // X tiles of head 0, head 1
  static constexpr uint32_t kOffW = kOffX + 2 * kBlk;   // weights [2][Q] fp32
  static constexpr uint32_t kOffBar = kOffW + 2 * Q * 4;
  static constexpr uint32_t kOffMisc = kOffBar + 2 * 8;
  // at NS = 256 at most two CTAs per SM, so that their TMEM columns fit the 512
  static constexpr uint32_t kNeed = kOffMisc + 16 + 1024;
  static constexpr uint32_t kBytes = NS == 256 && kNeed < 100 * 1024 ? 100 * 1024 : kNeed;
};

template <int Q, int NS, int kMode>
__global__ void __launch_bounds__(kThr) chunk_state_tc2_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                              const __grid_constant__ CUtensorMap tm_b,
                                                              const float* __restrict__ dA_cs,
                                                              const float* __restrict__ dt_c,
                                                              const float* __restrict__ phi, int64_t L, int64_t H,
                                                              int G, int64_t nc, int pairs_per_group,
                                                              float* __restrict__ states, int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  using S = TcSmem2<Q, NS>;
  constexpr uint32_t kBlkS = S::kBlk;
  const uint32_t bar_load = sbase + S::kOffBar, bar_mma = sbase + S::kOffBar + 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + S::kOffMisc);
  float* wsm = reinterpret_cast<float*>(gbase + S::kOffW);

  const int64_t c = blockIdx.x, b = blockIdx.z;
  const int g = (int)blockIdx.y / pairs_per_group, pr = (int)blockIdx.y % pairs_per_group;
  const int hpg = (int)(H / G);
  const int h0 = g * hpg + 2 * pr;
  const bool valid1 = 2 * pr + 1 < hpg;
  const int h1 = valid1 ? h0 + 1 : h0;
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_mbar_init();
  }
  // At NS = 16 the MMA runs over the whole zero-padded 64-column block.
  constexpr int kNm = NS < 64 ? 64 : NS;
  constexpr uint32_t kTm = kNm;  // TMEM columns
  if (warp == 0) {
    tmem_alloc(sbase + S::kOffMisc, kTm);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_load, (S::kNB + 2) * kBlkS);
    if (NS < 64) {
      tma_load_4d(sbase + S::kOffB, &tm_b, bar_load, 0, g, (int32_t)(c * Q), (int32_t)b);
    } else {
#pragma unroll
      for (int k = 0; k < NS / 64; ++k)
        tma_load_3d(sbase + S::kOffB + k * kBlkS, &tm_b, bar_load, g * NS + 64 * k, (int32_t)(c * Q), (int32_t)b);
    }
    tma_load_3d(sbase + S::kOffX, &tm_x, bar_load, h0 * kPs, (int32_t)(c * Q), (int32_t)b);
    tma_load_3d(sbase + S::kOffX + kBlkS, &tm_x, bar_load, h1 * kPs, (int32_t)(c * Q), (int32_t)b);
  }
  for (int e = tid; e < 2 * Q; e += kThr) {
    const int hh = e / Q, i = e % Q;
    const int64_t row = ((b * H + (hh ? h1 : h0)) * nc + c) * Q;
    const float cs_i = dA_cs[row + i];
    float w;
    if (kMode == 1) {
      w = expf(cs_i);
    } else {
      w = expf(dA_cs[row + Q - 1] - cs_i) * dt_c[row + i];
      if (kMode == 2) w *= cosf(phi[row + Q - 1] - phi[row + i]);
      if (kMode == 3) w *= sinf(phi[row + Q - 1] - phi[row + i]);
    }
    wsm[e] = w;
  }
  bool ok = __syncthreads_and(wait_bounded(bar_load, 0));
  if (ok) {
    for (int e = tid; e < 2 * Q; e += kThr) {
      const int hh = e / Q, r = e % Q;
      uint4* xt = reinterpret_cast<uint4*>(gbase + S::kOffX + hh * kBlkS);
      const float wv = wsm[e];
      const uint32_t wx = pack_bf16x2(wv, wv);
#pragma unroll
      for (uint32_t ch = 0; ch < 8; ++ch) {
        uint4 v = xt[sw128_offset((uint32_t)r, ch) >> 4];
        v.x = mul_bf16x2(v.x, wx);
        v.y = mul_bf16x2(v.y, wx);
        v.z = mul_bf16x2(v.z, wx);
        v.w = mul_bf16x2(v.w, wx);
        xt[sw128_offset((uint32_t)r, ch) >> 4] = v;
      }
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  if (ok && tid == 0) {
    tc_fence_after();
    constexpr uint32_t idesc = idesc_bf16_f32(128, kNm, 1, 1);  // X̃ᵀ (MN-major) · B (MN-major)
    const uint64_t da = smem_desc_sw128(sbase + S::kOffX, kBlkS, 1024);
    const uint64_t db = smem_desc_sw128(sbase + S::kOffB, kBlkS, 1024);
#pragma unroll
    for (uint32_t kk = 0; kk < Q / 16; ++kk) mma_ss(tmem, da + kk * 128u, db + kk * 128u, idesc, kk > 0);
    mma_commit(bar_mma);
  }
  if (ok) ok = wait_bounded(bar_mma, 0);
  ok = __syncthreads_and(ok);
  tc_fence_after();
  if (ok) {
    const uint32_t lane_addr = (32u * (uint32_t)warp) << 16;
    const int hh = tid >> 6, pp = tid & 63;
    float* dst = states + (((b * nc + c) * H + (hh ? h1 : h0)) * (int64_t)kPs + pp) * NS;
    if (NS == 16) {
      uint32_t r[16];
      tmem_ld16(tmem + lane_addr, r);
      tmem_ld_wait();
      reg_fence16(r);
      if (hh == 0 || valid1) {
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          d4[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]),
                              __uint_as_float(r[4 * e + 2]), __uint_as_float(r[4 * e + 3]));
      }
    }
#pragma unroll 1
    for (int q = 0; q < NS / 32; ++q) {
      uint32_t r[32];
      tmem_ld32(tmem + lane_addr + 32u * q, r);
      tmem_ld_wait();
      reg_fence(r);
      if (hh == 1 && !valid1) continue;
      float4* d4 = reinterpret_cast<float4*>(dst + 32 * q);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        d4[e] = make_float4(__uint_as_float(r[4 * e]), __uint_as_float(r[4 * e + 1]), __uint_as_float(r[4 * e + 2]),
                            __uint_as_float(r[4 * e + 3]));
    }
  }
  if (!ok && tid == 0 && err) atomicExch(err, (int32_t)SSD_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTm);
  }
}

}  // namespace

bool make_tma_map_bf16_narrow(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t G, int64_t N,
                              int box_rows) {
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
  if (!fn || N >= 64 || (N * 2) % 16 != 0) return false;
  cuuint64_t dims[4] = {(cuuint64_t)N, (cuuint64_t)G, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(N * 2), (cuuint64_t)(G * N * 2), (cuuint64_t)(L * G * N * 2)};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool chunk_state_tc_supported(const Problem& p) {
  return p.io == SSD_DTYPE_BF16 && p.P == kPs && (p.N == 16 || p.N == 64 || p.N == kNs || p.N == 256) &&
         (p.Q == 64 || p.Q == 128) && p.B > 0 && p.L > 0;
}

cudaError_t launch_chunk_state_tc(const Problem& p, int mode, const void* xin, const void* bin,
                                  const float* dA_cs, const float* dt_c, const float* phi, float* states,
                                  cudaStream_t s) {
  if (!chunk_state_tc_supported(p)) return cudaErrorNotSupported;
  CUtensorMap tx, tb;
  const bool narrow = p.N < 64;
  if (!make_tma_map_bf16(&tx, xin, p.B, p.L, p.H * kPs, (int)p.Q) ||
      !(narrow ? make_tma_map_bf16_narrow(&tb, bin, p.B, p.L, p.G, p.N, (int)p.Q)
               : make_tma_map_bf16(&tb, bin, p.B, p.L, p.G * p.N, (int)p.Q)))
    return cudaErrorInvalidValue;
  const int ppg = (int)(((p.H / p.G) + 1) / 2);
  dim3 grid((unsigned)p.nc, (unsigned)(p.G * ppg), (unsigned)p.B);
  auto launch = [&](auto kernel, uint32_t smem) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThr, smem, s>>>(tx, tb, dA_cs, dt_c, phi, p.L, p.H, (int)p.G, p.nc, ppg, states, p.err);
    return cudaGetLastError();
  };
  if (p.N != kNs) {
    auto run2 = [&](auto tag_q, auto tag_n) -> cudaError_t {
      constexpr int QQ = decltype(tag_q)::value, NN = decltype(tag_n)::value;
      constexpr uint32_t sm = TcSmem2<QQ, NN>::kBytes;
      switch (mode) {
        case 0: return launch(chunk_state_tc2_kernel<QQ, NN, 0>, sm);
        case 1: return launch(chunk_state_tc2_kernel<QQ, NN, 1>, sm);
        case 2: return launch(chunk_state_tc2_kernel<QQ, NN, 2>, sm);
        case 3: return launch(chunk_state_tc2_kernel<QQ, NN, 3>, sm);
        default: return cudaErrorInvalidValue;
      }
    };
    using I16 = std::integral_constant<int, 16>;
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    using I256 = std::integral_constant<int, 256>;
    if (p.Q == 128) return p.N == 16 ? run2(I128{}, I16{}) : p.N == 64 ? run2(I128{}, I64{}) : run2(I128{}, I256{});
    return p.N == 16 ? run2(I64{}, I16{}) : p.N == 64 ? run2(I64{}, I64{}) : run2(I64{}, I256{});
  }
  constexpr uint32_t s64 = TcSmem<64>::kBytes, s128 = TcSmem<128>::kBytes;
  const bool q128 = p.Q == 128;
  switch (mode) {
    case 0: return q128 ? launch(chunk_state_tc_kernel<128, 0>, s128) : launch(chunk_state_tc_kernel<64, 0>, s64);
    case 1: return q128 ? launch(chunk_state_tc_kernel<128, 1>, s128) : launch(chunk_state_tc_kernel<64, 1>, s64);
    case 2: return q128 ? launch(chunk_state_tc_kernel<128, 2>, s128) : launch(chunk_state_tc_kernel<64, 2>, s64);
    case 3: return q128 ? launch(chunk_state_tc_kernel<128, 3>, s128) : launch(chunk_state_tc_kernel<64, 3>, s64);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ssd
