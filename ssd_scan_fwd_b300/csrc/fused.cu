// fused.cu -- the whole SSD forward pass in one persistent kernel for
// sm_103a: TMA loads, tcgen05 tensor-core contractions with TMEM
// accumulators, the inter-chunk state kept on chip.
//
// Method (page "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of
// SSM)"): the recurrence h_t = α_t h_{t-1} + Δ_t B_t x_t, y_t = C_tᵀ h_t (+ D x_t)
// of §2.1.2/§2.1.1, evaluated chunk by chunk in the dual form of §2.2.1
// (Y = (L ⊙ C Bᵀ) X inside a chunk, mask L_ij = ∏_{k=j+1}^{i} α_k) with the
// state carried across chunks (block decomposition of the mask figure,
// §2.2.2).  For chunk k of one (batch b, head h), with cs the in-chunk
// running sum of log2 α (Δ·A·log2 e):
//   chunk_cumsum   cs_i and the per-chunk scalars                   (cumsum warp)
//   chunk_scan     S = C Bᵀ                                  (MMA, M=N=K=128)
//                  M_ij = S_ij 2^(cs_i − cs_j) Δ_j  (j ≤ i),
//                  plus D on the diagonal (the skip term D x_i)  (mask warpgroup → TMEM)
//                  Y = M X                                    (MMA, A from TMEM)
//                  Y_off = C h_inᵀ                            (MMA)
//                  y_i = Y_i + 2^cs_i Y_off,i                 (epilogue warpgroup)
//   chunk_state    S_cᵀ = Bᵀ (w ⊙ X), w_i = 2^(cs_last − cs_i) Δ_i   (MMA, M = N_state)
//   state_passing  h_in[k+1] = 2^cs_last h_in[k] + S_c        (epilogue, fp32 in registers)
//
// The mask is built in 32×32 blocks.  Below the diagonal block of its row
// quarter q (rows 32q..32q+31, reference token r = 32q) the decay factors
// split exactly: 2^(cs_i − cs_j) Δ_j = u_i · v_j with u_i = 2^(cs_i − cs_r) ≤ 1 and
// v_j = 2^(cs_r − cs_j) Δ_j ≤ Δ_j, so those blocks cost two multiplies per entry;
// only the four diagonal blocks evaluate an exponential per entry.
//
// Two heads of one group share a CTA: they share the C and B tiles and
// S = C Bᵀ, and their Y_off and S_c contractions run as single N = 128 MMAs.
// Layouts by instantiation: state size 128 (two heads, thread = state row n);
// 64, which also serves 16 with the C/B columns past 16 loaded as zeros (two
// heads, thread = state row (head, p), S_c = [X̃_0 | X̃_1]ᵀ B); 256 (one head
// per CTA, the two head warpgroups splitting its state rows, mask column
// blocks, X̃ rows and y columns); the complex decay at 128 (one head per CTA,
// the Re / Im parts of its state in the places of the two heads, the two
// warpgroups splitting the state's columns p); the retrieval rank (rows
// (token, rank), the token's Δ and decay shared by its R rows).  The one-head
// and 64-column layouts give the control warpgroup 144 registers and the
// head warpgroups 176 (setmaxnreg).
//
// Work units.  A unit is a run of consecutive chunks of the sequence (nc
// chunks) of a head pair of one batch row.  It starts from the state its
// predecessor published in the workspace (flag + fp32 state), or from
// init_state at chunk 0; a unit that ends the sequence writes final_state.
// With at least as many sequences as CTAs, the sequences laid end to end are
// cut into one contiguous range per CTA (cta_unit): every CTA gets the same
// number of chunks and hands a state off at most once.  Otherwise each
// sequence is cut into nseg segments, numbered segment-major and dealt
// round-robin (the two-pass mode publishes every segment's entering state
// before the kernel starts).
//
// Warp roles (384 threads, one CTA per SM):
//   warp 0      TMA producers: lane 0 loads the C and B tiles (released once
//               the MMAs reading them are issued and done), lanes 1-2 the X
//               tiles of each head (2-stage rings, released after y is stored);
//               lane 3 raises the segment flags; lane 4 issues the TMA
//               stores of y
//   warp 1      TMEM allocator and MMA issuer (one thread): four in-order
//               streams -- S(k), Y_off(k), S_c(k), Y(k) -- each op issued as soon
//               as its inputs are ready
//   warps 2, 3  chunk_cumsum of Δ·A and the per-chunk scalars, one head each
//   warps 4-7   head 0, warps 8-11 head 1: X̃ = w ⊙ X, the decay mask
//               (thread = row), the state update (thread = state row n), the y
//               epilogue (thread = token row i), segment hand-off
// TMEM (512 columns): S 128, masks 2×64 (bf16 pairs), Y_off 128 (both
// heads), S_c 128 (both heads; Y takes its columns once the state updates
// have read it, so S of the next chunk never waits for the y epilogue).
// Every wait is bounded: on timeout the CTA raises an abort flag, records
// SSD_ERR_TIMEOUT in the workspace word, drains what it issued and exits.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "sm100.cuh"

namespace ssd {
namespace {

using namespace sm100;

constexpr int kQ = 128;  // chunk length (tokens)
constexpr int kP = 64;   // head dim
constexpr int kN = 128;  // state dim of the two-pass segment-state kernels
constexpr int kThreads = 384;

// ---- shared memory layout (offsets from a 1024-byte aligned base) ----
constexpr uint32_t kBlk = kQ * 128;       // one [128 rows][128 B] swizzled block
constexpr int kXStages = 2;               // X ring depth per head
// scalar block (floats): cs2[128] u[128] ej[128] w[128] ecs[128] v[192] decay
constexpr int SC_CS2 = 0, SC_U = 128, SC_EJ = 256, SC_W = 384, SC_ECS = 512, SC_V = 640, SC_DECAY = 832;
constexpr uint32_t kScalHead = 864 * 4;
// complex decay (one head per CTA) adds: the imaginary weights wi[128] (bf16
// pairs), cos φ[128], sin φ[128], v ⊙ sin φ [192] (SC_V then holds v ⊙ cos φ)
// and the imaginary part of the chunk decay
constexpr int SC_WI = 864, SC_CPH = 992, SC_SPH = 1120, SC_VS = 1248, SC_DECAY_IM = 1440;
constexpr uint32_t kScalHeadRot = 1444 * 4;
constexpr uint32_t kScalSlot = 2 * kScalHead;
constexpr int kScalSlots = 4;  // scalar ring depth: the cumsum warp runs up to three chunks ahead

enum : uint32_t {
  B_CBF = 0, B_CBE,                            // C/B tiles landed / MMAs done with them
  B_XF00, B_XF01, B_XF10, B_XF11,              // X ring [head][stage]: TMA landed
  B_XE00, B_XE01, B_XE10, B_XE11,              // X ring [head][stage]: y stored from it
  B_CSF0, B_CSF1, B_CSF2, B_CSF3,              // scalar ring [slot]: written
  B_CSE0, B_CSE1, B_CSE2, B_CSE3,              // scalar ring [slot]: read by both head warpgroups
  B_SFULL,                                     // S(k) in TMEM
  B_SYEMPTY,                                   // Y(k), Y_off(k) read back
  B_MFULL0, B_MFULL1, B_MEMPTY,                // masks [head] in TMEM / Y(k) done with them
  B_XTFULL, B_XTEMPTY,                         // X̃(k) written / S_c(k) done with it
  B_HFULL, B_HEMPTY,                           // bf16 states in smem / Y_off done with them
  B_SCFULL, B_SCEMPTY,                         // chunk states in TMEM / read
  B_YFULL, B_YOFFFULL,                         // Y(k) / Y_off(k) in TMEM
  B_YST00, B_YST01, B_YST10, B_YST11,          // y staged in X[head][stage] for the TMA store
  B_PUB0, B_PUB1,                              // segment state of head h stored
  B_PUBACK,                                    // the flags of a hand-off are raised
  B_ZF,                                        // gate: z tiles of both heads in the X̃ blocks
  B_ZE0, B_ZE1,                                // gate: head h's warpgroup has read its z tile
  B_DRAIN,
  kBarCount
};
// Shared memory of the fused kernel for state size NS (128, or 64: the 64
// columns also serve dstate 16, whose C/B columns past 16 load as zeros).
template <int NS, bool kRot = false>
struct Lay {
  static constexpr uint32_t kNB = NS / 64;                          // 64-column blocks of a C or B tile
  static constexpr uint32_t kHeads = (NS == 256 || kRot) ? 1 : 2;   // heads per CTA
  static constexpr uint32_t kXtBlocks = kRot ? 2 : kHeads;          // X̃ blocks: per head, or Re / Im of the one head
  static constexpr uint32_t kOffC = 0;                              // C tile: kNB blocks
  static constexpr uint32_t kOffB = kNB * kBlk;                     // B tile: kNB blocks
  static constexpr uint32_t kCBBytes = 2 * kNB * kBlk;
  static constexpr uint32_t kOffX = kCBBytes;                       // X tiles [head][stage] (also the y staging tiles)
  static constexpr uint32_t kOffXt = kOffX + kHeads * kXStages * kBlk;  // X̃ = w ⊙ X: [head] blocks
  static constexpr uint32_t kOffHb = kOffXt + kXtBlocks * kBlk;     // bf16 carried states
  // NS = 128: [head] blocks [n][p] (MN-major B operand of Y_off);
  // NS = 64: one block [(head, p)][n] (K-major B operand of Y_off);
  // NS = 256: blocks [n half][n][p] of the one head (MN-major);
  // complex decay: blocks [Re / Im][n][p] of the one head (MN-major)
  static constexpr uint32_t kHbBytes = (NS == 64 ? 1 : 2) * kBlk;
  static constexpr uint32_t kScalHeadBytes = kRot ? kScalHeadRot : kScalHead;
  static constexpr uint32_t kScalSlotBytes = kHeads * kScalHeadBytes;  // scalars of one chunk: [head]
  static constexpr uint32_t kOffScal = kOffHb + kHbBytes;           // per-chunk scalars: [slot][head]
  static constexpr uint32_t kOffBar = kOffScal + kScalSlots * kScalSlotBytes;
  static constexpr uint32_t kOffMisc = kOffBar + kBarCount * 8;     // tmem base, abort flag
  static constexpr uint32_t kSmemAlloc = kOffMisc + 16 + 1024;
  static_assert(kSmemAlloc <= 232448, "shared memory budget");
};

// ---- TMEM columns (fp32 accumulators, lane = row) ----
constexpr uint32_t kTmS = 0;       // S(k) = C Bᵀ, 128 columns
constexpr uint32_t kTmMK = 128;    // masks, bf16 pairs: head h in 128 + 64h
constexpr uint32_t kTmYoff = 256;  // Y_off = C [h_0ᵀ | h_1ᵀ]: head h in 256 + 64h
constexpr uint32_t kTmSc = 384;    // S_cᵀ = Bᵀ [X̃_0 | X̃_1]: head h in 384 + 64h; once the state
                                   // update has read it, Y_h = M_h X_h in the same columns
constexpr uint32_t kTmCols = 512;

constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, 0, 0);     // C (K-major) · Bᵀ (K-major)
constexpr uint32_t kIdescYoff = idesc_bf16_f32(128, 128, 0, 1);  // C (K-major) · [h_0ᵀ | h_1ᵀ] (MN-major)
constexpr uint32_t kIdescSc = idesc_bf16_f32(128, 128, 1, 1);    // Bᵀ (MN-major) · [X̃_0 | X̃_1] (MN-major)
constexpr uint32_t kIdescY = idesc_bf16_f32(128, 64, 0, 1);      // M_h (TMEM) · X_h (MN-major)
// state size 64: S_c = [X̃_0 | X̃_1]ᵀ B (M = both heads' rows p, N = 64 state
// columns; both operands MN-major), Y_off = C [h_0 | h_1]ᵀ with the states
// stored [(head, p)][n] (K-major)
constexpr uint32_t kIdescSc64 = idesc_bf16_f32(128, 64, 1, 1);
constexpr uint32_t kIdescYoff64 = idesc_bf16_f32(128, 128, 0, 0);

struct FusedParams {
  const float* dt;
  const float* A;
  const float* D;
  const float* init;
  float* final_state;
  int32_t B, L, H, G, nc;
  int32_t pairs_per_group;  // sequences per group: ceil((H/G) / 2) head pairs, or H/G single heads
  int32_t chains;           // B · G · pairs_per_group: sequences of head pairs (or heads)
  int32_t heads_per_chain;  // 2 (state sizes 64, 128) or 1 (state size 256)
  int32_t nseg;             // segments per sequence (round-robin schedule); 1 for ranges
  int32_t units;            // chains · nseg
  int32_t ranges;           // 1: contiguous chunk ranges per CTA (see cta_unit), 0: round-robin units
  int32_t* err;             // workspace word: SSD_ERR_TIMEOUT on a timed-out wait
  uint32_t* seg_flag;       // [B·H][nseg]: 1 once the segment's end state of a head is published
  float* seg_state;         // [B·H][nseg][P][N] fp32
  uint64_t timeout_ns;
  long long* trace;         // optional per-chunk role timestamps of CTA 0 (SSD_FUSED_TRACE)
  int32_t publish;          // 0: entering states were published beforehand (two-pass mode)
  const float* dt_bias;     // [H] or null: Δ = dt + dt_bias (instantiations with kDelta)
  int32_t dt_softplus;      // 1: Δ = softplus(dt + dt_bias)
  int32_t test_no_flags;    // test of the bounded waits: hand-off flags are never raised
  int32_t nstate;           // N of the problem (NS = 64 also serves N = 16)
  int32_t Ltok;             // tokens per batch row (L counts rows: Ltok << rank_log2)
  int32_t rank_log2;        // retrieval rank R = 2^rank_log2: the R rows of a token share its decay
  int32_t narrow;           // 1: C/B tensor maps are the 4-D narrow ones (N < 64, columns past N read as 0)
  int32_t pdl;              // 1: launched as a programmatic dependent of the segment-combine kernel
  uint32_t zero_words;      // two-pass mode: 16-byte words at err (status word, flags) the states kernel clears
  const float* theta;       // complex decay: rotation angle per token and head, [B][L][H]
  const float* init_im;     // complex decay: imaginary part of init_state (or null)
  float* final_im;          // complex decay: imaginary part of final_state (or null)
};

// Trace events (SM clock, CTA 0, first kTraceChunks chunks): one row of
// kTraceEvents per chunk.  Head 0's warpgroup records its own phases.
constexpr int kTraceChunks = 64, kTraceEvents = 16;
constexpr int kTraceCtas = 256;  // per-CTA [start ns, end ns, chunks, SM, start clock, end clock] follow the chunk rows
enum : int {
  E_PROD = 0, E_CS, E_MMA_YOFF, E_MMA_SC, E_MMA_S, E_MMA_Y, E_XT_START, E_XT_END, E_MK3_START, E_MK3_END,
  E_ST_START, E_ST_END, E_Y_START, E_Y_END, E_STORE, E_MK0_END
};

__device__ __forceinline__ void trace_ev(const long long* base, uint32_t k, int ev) {
  if (base != nullptr && blockIdx.x == 0 && k < (uint32_t)kTraceChunks)
    const_cast<long long*>(base)[k * kTraceEvents + ev] = clock64();
}

// One work unit: the chunks [c0, c1) of the sequence of a head pair (h[0],
// h[1]) of one batch row.  When the group has an odd number of heads, its
// last pair has one real head: h[1] repeats h[0] and nothing of it is
// written (valid1).  The unit starts from init_state (or zero) when `first`,
// else from the state published in slot `pred`; it writes final_state when
// `last`, else publishes its leaving state in slot `pub`.
struct Unit {
  int b, g, s, c0, c1;
  int h[2];
  bool valid1, first, last;
  int pred, pub;
};

__device__ __forceinline__ void chain_info(const FusedParams& p, int chain, Unit& w) {
  const int per_b = p.G * p.pairs_per_group;
  w.b = chain / per_b;
  const int rem = chain - w.b * per_b;
  w.g = rem / p.pairs_per_group;
  const int pr = rem - w.g * p.pairs_per_group;
  const int hpg = p.H / p.G;
  w.h[0] = w.g * hpg + p.heads_per_chain * pr;
  w.valid1 = p.heads_per_chain == 2 && 2 * pr + 1 < hpg;
  w.h[1] = w.valid1 ? w.h[0] + 1 : w.h[0];
}

// Round-robin schedule: unit u is segment s = u / chains of sequence
// u % chains (segment-major), dealt to CTA u % gridDim.x.
__device__ __forceinline__ Unit unit_info(const FusedParams& p, int u) {
  Unit w;
  w.s = u / p.chains;
  chain_info(p, u - w.s * p.chains, w);
  w.c0 = (int)((int64_t)w.s * p.nc / p.nseg);
  w.c1 = (int)((int64_t)(w.s + 1) * p.nc / p.nseg);
  w.first = w.s == 0;
  w.last = w.s == p.nseg - 1;
  w.pred = w.s - 1;
  w.pub = w.s;
  return w;
}

// The j-th unit of this CTA, in processing order; false past the last one.
// Every unit has at least one chunk.
//
// Contiguous ranges (at least as many sequences as CTAs): the chunks of all
// sequences, laid end to end sequence after sequence, are cut into gridDim.x
// equal ranges, one per CTA.  A range is at least one sequence long, so it
// holds the tail of one sequence, whole sequences, and the head of another;
// a CTA takes its sequences from the last to the first.  The head piece of a
// sequence (from chunk 0) is then its CTA's first unit and the tail piece
// its neighbour's last, so the tail's entering state is published about a
// range length minus a sequence length before it is needed, and a CTA hands
// off at most once in each direction.
__device__ __forceinline__ bool cta_unit(const FusedParams& p, int j, Unit& w) {
  if (!p.ranges) {
    const int u = (int)blockIdx.x + j * (int)gridDim.x;
    if (u >= p.units) return false;
    w = unit_info(p, u);
    return true;
  }
  const int64_t total = (int64_t)p.chains * p.nc;
  const int64_t s = (int64_t)blockIdx.x * total / gridDim.x;
  const int64_t e = (int64_t)(blockIdx.x + 1) * total / gridDim.x;
  const int64_t x = (e - 1) / p.nc - j;
  if (e <= s || x < s / p.nc) return false;
  chain_info(p, (int)x, w);
  const int64_t base = x * p.nc;
  w.c0 = (int)((s > base ? s : base) - base);
  w.c1 = (int)((e < base + p.nc ? e : base + p.nc) - base);
  w.first = w.c0 == 0;
  w.last = w.c1 == p.nc;
  w.s = w.first ? 0 : 1;
  w.pred = 0;
  w.pub = 0;
  return true;
}

// Walks the chunks of the units a CTA owns, in order.
struct Cursor {
  int j, c;
  bool ok;
  uint32_t k;  // chunks walked so far
  Unit w;
  __device__ __forceinline__ void start(const FusedParams& p) {
    j = 0;
    k = 0;
    ok = cta_unit(p, 0, w);
    if (ok) c = w.c0;
  }
  __device__ __forceinline__ bool live() const { return ok; }
  __device__ __forceinline__ void next(const FusedParams& p) {
    ++k;
    if (++c >= w.c1) {
      ok = cta_unit(p, ++j, w);
      if (ok) c = w.c0;
    }
  }
};

struct Ctl {
  volatile uint32_t* abort;
  int32_t* err;
  uint64_t timeout;
};

__device__ __forceinline__ void raise_abort(const Ctl& c) {
  *c.abort = 1u;
  if (c.err) atomicExch(c.err, (int32_t)SSD_ERR_TIMEOUT);
}

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
      raise_abort(c);
      return false;
    }
  }
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh by the hardware's approximation (PTX tanh.approx.f32, relative error
// about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// silu(z) = z σ(z) = h (1 + tanh h), h = z / 2: one MUFU operation and one
// FMA (the division form takes two MUFU operations, and the MUFU pipe sets
// the pace of the gated y epilogue).  Absolute error ≤ |z| 2^-12: below the
// bf16 rounding of the gated output for z ≥ −2; for z < −2, where silu is
// small, it is an absolute error, not a relative one.
__device__ __forceinline__ float silu(float z) {
  const float h = 0.5f * z;
  return fmaf(h, tanh_approx(h), h);
}

// softplus(v) = log(1 + e^v) = max(v, 0) + log1p(t), t = e^{-|v|} ∈ (0, 1].
// log1p(t) = ln(u) · t / (u − 1) with u = 1 + t rounded (u − 1 is exact, and
// this rearrangement, Goldberg's, keeps the relative accuracy of ln for small
// t), and t itself when u rounds to 1.  Relative error a few 1e-6.
__device__ __forceinline__ float softplus(float v) {
  const float t = ex2(-1.4426950408889634f * fabsf(v));
  const float u = 1.f + t;
  const float d = u - 1.f;
  float lg;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lg) : "f"(u));
  const float l1p = d == 0.f ? t : 0.6931471805599453f * lg * __fdividef(t, d);
  return fmaxf(v, 0.f) + l1p;
}

// Eight K=16 MMAs of one K=128 contraction.  Operand descriptors are built
// once; each step adds a constant to the start-address field (16-byte units):
// operands whose K is the state dimension (two 64-wide column blocks) advance
// 32 bytes within a block and jump a block every 4 steps; operands whose K is
// the 128 token rows (128 bytes each) advance 16 rows = 2048 bytes.
enum : int { KSTEP_COLS = 0, KSTEP_ROWS = 1 };

template <int KA, int KB, int STEPS = 8>
__device__ __forceinline__ void mma_k128_ss(uint32_t d, uint64_t da, uint64_t db, uint32_t idesc) {
#pragma unroll
  for (uint32_t kk = 0; kk < STEPS; ++kk) {
    const uint64_t oa = KA == KSTEP_COLS ? (uint64_t)((kk >> 2) * (kBlk >> 4) + (kk & 3u) * 2u) : (uint64_t)(kk * 128u);
    const uint64_t ob = KB == KSTEP_COLS ? (uint64_t)((kk >> 2) * (kBlk >> 4) + (kk & 3u) * 2u) : (uint64_t)(kk * 128u);
    mma_ss(d, da + oa, db + ob, idesc, kk > 0);
  }
}

__device__ __forceinline__ void mma_k128_ts(uint32_t d, uint32_t ta, uint64_t db, uint32_t idesc) {
#pragma unroll
  for (uint32_t kk = 0; kk < 8; ++kk) mma_ts(d, ta + kk * 8u, db + (uint64_t)(kk * 128u), idesc, kk > 0);
}

template <int NS>
__device__ __forceinline__ uint32_t x_tile(uint32_t head, uint32_t k) {
  return Lay<NS>::kOffX + (head * kXStages + (k % kXStages)) * kBlk;
}

// kDelta: Δ = [softplus](dt + dt_bias) formed by the cumsum warps.  kGate:
// y ← y · silu(z); the MMA thread loads the z tiles of chunk k into the X̃
// blocks once S_c(k) has read X̃(k), and the head warpgroups read them in the
// y epilogue, before they write X̃(k+1).  kRank: retrieval rank R > 1 (rows
// are (token, rank) pairs; p.rank_log2 read at run time).  kRot: complex
// decay α_t = e^{Δ_t A}(cos θ_t + i sin θ_t) at state size 128, one head per
// CTA: the Re / Im parts of the state take the places of the two heads in
// X̃ (two weightings of X), S_c and Y_off, and the two warpgroups split the
// state's columns p.  Separate instantiations, so that the plain forward
// pass carries none of it.
template <bool kDelta, bool kGate, int NS, bool kRank = false, bool kRot = false>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_fused_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
                     const __grid_constant__ CUtensorMap tm_z, const FusedParams p) {
  static_assert(!kRot || (NS == 128 && !kDelta && !kGate && !kRank), "complex decay: state size 128, plain pass");
  using L = Lay<NS, kRot>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](uint32_t i) { return sbase + L::kOffBar + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + L::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + L::kOffMisc + 4);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    uint32_t counts[kBarCount];
    for (uint32_t i = 0; i < kBarCount; ++i) counts[i] = 1;  // TMA expect_tx, MMA commits, store warp
    for (int i = 0; i < kScalSlots; ++i) {
      counts[B_CSF0 + i] = 32 * L::kHeads;                    // the cumsum warps (one per head)
      counts[B_CSE0 + i] = 256;                               // both head warpgroups
    }
    counts[B_SYEMPTY] = counts[B_XTFULL] = counts[B_HFULL] = counts[B_SCEMPTY] = 256;
    counts[B_MFULL0] = counts[B_MFULL1] = 128;                // one head warpgroup each
    counts[B_YST00] = counts[B_YST01] = counts[B_YST10] = counts[B_YST11] = 128;
    counts[B_PUB0] = counts[B_PUB1] = 128;
    counts[B_ZE0] = counts[B_ZE1] = 128;
    for (uint32_t i = 0; i < kBarCount; ++i) mbar_init(bar(i), counts[i]);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + L::kOffMisc, kTmCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    tma_prefetch_desc(&tm_c);
    tma_prefetch_desc(&tm_y);
    if constexpr (kGate) tma_prefetch_desc(&tm_z);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas) {
    long long* t = const_cast<long long*>(p.trace) + kTraceChunks * kTraceEvents + 6 * blockIdx.x;
    t[0] = (long long)globaltimer_ns();
    t[4] = clock64();
  }

  // Register budgets per warpgroup, one role-independent call per warpgroup
  // before its roles branch: the control warpgroup (warps 0-3) hands
  // registers back, the two head warpgroups take them (128 × 144 + 256 × 176
  // = 63488 of the 384 × 168 = 64512 the block is launched with).  Not at
  // state size 128 with real decay, which measured as fast or faster without.
  constexpr bool kBudget = NS != 128 || kRot;
  if (warp < 4) {
  if constexpr (kBudget) setmaxnreg_dec<144>();
  if (warp == 0 && lane == 3) {
    // ------------------------------------------------------------ segment flags
    // For every unit of this CTA that ends before the last segment: once both
    // head warpgroups have stored their state rows and arrived, make the
    // stores visible at GPU scope and raise the heads' flags.
    uint32_t npub = 0;
    Unit w;
    for (int j = 0; p.publish && cta_unit(p, j, w); ++j) {
      if (w.last) continue;
      if (!wait_bar(bar(B_PUB0), npub & 1u, ctl) || !wait_bar(bar(B_PUB1), npub & 1u, ctl)) break;
      __threadfence();
      if (!p.test_no_flags) {
        st_release_u32(p.seg_flag + ((int64_t)w.b * p.H + w.h[0]) * p.nseg + w.pub, 1u);
        if (w.valid1) st_release_u32(p.seg_flag + ((int64_t)w.b * p.H + w.h[1]) * p.nseg + w.pub, 1u);
      }
      mbar_arrive(bar(B_PUBACK));
      ++npub;
    }
  } else if (warp == 0 && lane == 4) {
    // ------------------------------------------------------------ y stores, both heads
    {
      // y is not read again (an eviction hint only in the one-head layouts,
      // where it measured faster; the two-head layout is faster without)
      constexpr bool kHint = NS == 256 || kRot;
      const uint64_t pol_y = kHint ? l2_policy_evict_first() : 0ull;
      uint32_t k = 0;
      bool ok = true;
      Unit w;
      for (int j = 0; ok && cta_unit(p, j, w); ++j) {
        for (int c = w.c0; c < w.c1 && ok; ++c, ++k) {
          const uint32_t s = k % kXStages, ph = (k / kXStages) & 1u;
          for (uint32_t hh = 0; hh < 2; ++hh) {
            if (!(ok = wait_bar(bar(B_YST00 + 2 * hh + s), ph, ctl))) break;
            if (hh == 0) trace_ev(p.trace, k, E_STORE);
            // at state size 256 both warpgroups stage halves of the one head's
            // tile: it is stored once both have arrived
            const uint32_t th = L::kHeads == 1 ? 0u : hh;
            if ((L::kHeads == 1 && hh == 1) || (L::kHeads == 2 && (hh == 0 || w.valid1))) {
              if constexpr (kHint)
                tma_store_3d_hint(&tm_y, sbase + x_tile<NS>(th, k), (th ? w.h[1] : w.h[0]) * kP, c * kQ, w.b, pol_y);
              else
                tma_store_3d(&tm_y, sbase + x_tile<NS>(th, k), (th ? w.h[1] : w.h[0]) * kP, c * kQ, w.b);
              tma_store_commit();
            }
          }
          if (!ok) break;
          tma_store_wait_read0();
          mbar_arrive(bar(B_XE00 + s));
          mbar_arrive(bar(B_XE10 + s));
        }
      }
      tma_store_wait_all0();
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producers
    // lane 0: C and B tiles (single stage, released once S, Y_off and S_c of
    // the chunk are done); lanes 1, 2: X tiles of head 0 / 1 (2-stage rings,
    // released after y has been stored from them).
    if (lane < 1 + (int)L::kHeads) {
      // one-head layouts: C and B tiles are read by every head's CTA of the
      // group (kept in L2), x once (evicted first); the two-head layout
      // measured faster without the hints
      constexpr bool kHint = NS == 256 || kRot;
      const uint64_t pol = !kHint ? 0ull : lane == 0 ? l2_policy_evict_last() : l2_policy_evict_first();
      uint32_t k = 0;
      bool ok = true;
      Unit w;
      for (int j = 0; ok && cta_unit(p, j, w); ++j) {
        for (int c = w.c0; c < w.c1; ++c, ++k) {
          if (lane == 0) {
            if (!(ok = wait_bar(bar(B_CBE), (k & 1u) ^ 1u, ctl))) break;
            trace_ev(p.trace, k, E_PROD);
            mbar_arrive_expect_tx(bar(B_CBF), L::kCBBytes);
            if (p.narrow) {  // [B][L][G][N] maps, one 64-column box zero-filled past N
              tma_load_4d(sbase + L::kOffC, &tm_c, bar(B_CBF), 0, w.g, c * kQ, w.b);
              tma_load_4d(sbase + L::kOffB, &tm_b, bar(B_CBF), 0, w.g, c * kQ, w.b);
            } else {
#pragma unroll
              for (uint32_t nb = 0; nb < L::kNB; ++nb) {
                if constexpr (kHint) {
                  tma_load_3d_hint(sbase + L::kOffC + nb * kBlk, &tm_c, bar(B_CBF), w.g * NS + 64 * nb, c * kQ, w.b,
                                   pol);
                  tma_load_3d_hint(sbase + L::kOffB + nb * kBlk, &tm_b, bar(B_CBF), w.g * NS + 64 * nb, c * kQ, w.b,
                                   pol);
                } else {
                  tma_load_3d(sbase + L::kOffC + nb * kBlk, &tm_c, bar(B_CBF), w.g * NS + 64 * nb, c * kQ, w.b);
                  tma_load_3d(sbase + L::kOffB + nb * kBlk, &tm_b, bar(B_CBF), w.g * NS + 64 * nb, c * kQ, w.b);
                }
              }
            }
          } else {
            const uint32_t hh = lane - 1, s = k % kXStages, ph = (k / kXStages) & 1u;
            if (!(ok = wait_bar(bar(B_XE00 + 2 * hh + s), ph ^ 1u, ctl))) break;
            mbar_arrive_expect_tx(bar(B_XF00 + 2 * hh + s), kBlk);
            if constexpr (kHint)
              tma_load_3d_hint(sbase + x_tile<NS>(hh, k), &tm_x, bar(B_XF00 + 2 * hh + s), (hh ? w.h[1] : w.h[0]) * kP,
                               c * kQ, w.b, pol);
            else
              tma_load_3d(sbase + x_tile<NS>(hh, k), &tm_x, bar(B_XF00 + 2 * hh + s), (hh ? w.h[1] : w.h[0]) * kP,
                          c * kQ, w.b);
          }
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA exits
        const uint32_t depth = lane == 0 ? 1u : (uint32_t)kXStages;
        for (uint32_t j = (k >= depth ? k - depth : 0); j < k; ++j) {
          const uint32_t b2 = lane == 0 ? bar(B_CBF) : bar(B_XF00 + 2 * (lane - 1) + j % kXStages);
          const uint32_t par = lane == 0 ? (j & 1u) : ((j / kXStages) & 1u);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(b2, par) && globaltimer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t total = 0;  // chunks this CTA processes
      {
        Unit w;
        for (int j = 0; cta_unit(p, j, w); ++j) total += (uint32_t)(w.c1 - w.c0);
      }
      // Operand descriptors, built once.
      const uint64_t dC = smem_desc_sw128(sbase + L::kOffC, 16, 1024);
      const uint64_t dBk = smem_desc_sw128(sbase + L::kOffB, 16, 1024);
      const uint64_t dBm = smem_desc_sw128(sbase + L::kOffB, kBlk, 1024);
      const uint64_t dH = smem_desc_sw128(sbase + L::kOffHb, kBlk, 1024);
      const uint64_t dXt = smem_desc_sw128(sbase + L::kOffXt, kBlk, 1024);
      const uint64_t dX = smem_desc_sw128(sbase + L::kOffX, kBlk, 1024);
      const uint64_t dHk = smem_desc_sw128(sbase + L::kOffHb, 16, 1024);  // NS = 64: [(head, p)][n]
      // Next op of each stream: S(kS), Y_off(kO), S_c(kC), Y(kY).  The C/B
      // tiles of chunk k are released once S(k), Y_off(k) and S_c(k) are issued.
      uint32_t kS = 0, kO = 0, kC = 0, kY = 0;
      Cursor zc;  // gate: chunk whose z tiles are loaded next
      if constexpr (kGate) zc.start(p);
      uint64_t t_idle = globaltimer_ns();
      bool ok = true;
      while (ok && (kS < total || kO < total || kC < total || kY < total || (kGate && zc.live()))) {
        bool progress = false;
        // The checks run in the order of the chain S -> masks -> Y -> y that sets
        // the pace (an issuing thread waits while the tensor pipe is busy):
        // S, Y, then S_c and Y_off, which are needed later in the chunk.
        // ---- S(k) = C Bᵀ, once both masks of chunk k-1 have read S(k-1)
        if (kS < total) {
          const uint32_t k = kS;
          if (mbar_test_wait(bar(B_CBF), k & 1u) && mbar_test_wait(bar(B_MFULL0), (k & 1u) ^ 1u) &&
              mbar_test_wait(bar(B_MFULL1), (k & 1u) ^ 1u)) {
            trace_ev(p.trace, k, E_MMA_S);
            tc_fence_after();
            mma_k128_ss<KSTEP_COLS, KSTEP_COLS, NS / 16>(tmem + kTmS, dC, dBk, kIdescS);
            mma_commit(bar(B_SFULL));
            ++kS;
            if (kO >= kS && kC >= kS) mma_commit(bar(B_CBE));
            progress = true;
          }
        }
        // ---- Y_h(k) = M_h X_h into the S_c columns of head h, once both state
        // updates have read S_c(k);
        // A = mask from TMEM (bf16 pairs, 8 columns per K = 16), B = X MN-major
        if (kY < kS) {
          const uint32_t k = kY, xs = k % kXStages, xph = (k / kXStages) & 1u;
          if (mbar_test_wait(bar(B_MFULL0), k & 1u) && mbar_test_wait(bar(B_MFULL1), k & 1u) &&
              mbar_test_wait(bar(B_SCEMPTY), k & 1u) && mbar_test_wait(bar(B_XF00 + xs), xph) &&
              (L::kHeads == 1 || mbar_test_wait(bar(B_XF10 + xs), xph))) {
            trace_ev(p.trace, k, E_MMA_Y);
            tc_fence_after();
            mma_k128_ts(tmem + kTmSc, tmem + kTmMK, dX + (uint64_t)(xs * (kBlk >> 4)), kIdescY);
            if (L::kHeads == 2)
              mma_k128_ts(tmem + kTmSc + 64u, tmem + kTmMK + 64u,
                          dX + (uint64_t)((kXStages + xs) * (kBlk >> 4)), kIdescY);
            mma_commit(bar(B_YFULL));
            mma_commit(bar(B_MEMPTY));
            ++kY;
            progress = true;
          }
        }
        // ---- S_cᵀ(k) = Bᵀ [X̃_0 | X̃_1]: A = B tile read MN-major (M = state rows
        // in two 64-wide atoms), B = X̃ MN-major (N = 2·P); K = token rows.
        if (kC < total) {
          const uint32_t k = kC;
          if (mbar_test_wait(bar(B_CBF), k & 1u) && mbar_test_wait(bar(B_XTFULL), k & 1u) &&
              mbar_test_wait(bar(B_SYEMPTY), (k & 1u) ^ 1u)) {
            trace_ev(p.trace, k, E_MMA_SC);
            tc_fence_after();
            if constexpr (NS == 128) {
              mma_k128_ss<KSTEP_ROWS, KSTEP_ROWS>(tmem + kTmSc, dBm, dXt, kIdescSc);
            } else if constexpr (NS == 64) {
              mma_k128_ss<KSTEP_ROWS, KSTEP_ROWS>(tmem + kTmSc, dXt, dBm, kIdescSc64);
            } else {
              // one head: S_cᵀ of state rows n in [0, 128) and [128, 256), A = the
              // B tile's blocks (2g, 2g+1) read MN-major, B = X̃ (N = P)
              mma_k128_ss<KSTEP_ROWS, KSTEP_ROWS>(tmem + kTmSc, dBm, dXt, kIdescSc64);
              mma_k128_ss<KSTEP_ROWS, KSTEP_ROWS>(tmem + kTmSc + 64u, dBm + (uint64_t)((2 * kBlk) >> 4), dXt,
                                                  kIdescSc64);
            }
            mma_commit(bar(B_SCFULL));
            mma_commit(bar(B_XTEMPTY));
            ++kC;
            if (kS >= kC && kO >= kC) mma_commit(bar(B_CBE));
            progress = true;
          }
        }
        // ---- Y_off(k) = C [h_0ᵀ | h_1ᵀ]: states stored [n][p] per head, MN-major, K = n.
        // Its TMEM columns are free once Y_off(k-1) has been read back.
        if (kO < total) {
          const uint32_t k = kO;
          if (mbar_test_wait(bar(B_CBF), k & 1u) && mbar_test_wait(bar(B_HFULL), k & 1u) &&
              mbar_test_wait(bar(B_SYEMPTY), (k & 1u) ^ 1u)) {
            trace_ev(p.trace, k, E_MMA_YOFF);
            tc_fence_after();
            if constexpr (NS == 128)
              mma_k128_ss<KSTEP_COLS, KSTEP_ROWS>(tmem + kTmYoff, dC, dH, kIdescYoff);
            else if constexpr (NS == 64)
              mma_k128_ss<KSTEP_COLS, KSTEP_COLS, 4>(tmem + kTmYoff, dC, dHk, kIdescYoff64);
            else  // one head: K = 256 state rows of [n][p] (two blocks, contiguous), N = P
              mma_k128_ss<KSTEP_COLS, KSTEP_ROWS, 16>(tmem + kTmYoff, dC, dH, kIdescY);
            mma_commit(bar(B_YOFFFULL));
            mma_commit(bar(B_HEMPTY));
            ++kO;
            if (kS >= kO && kC >= kO) mma_commit(bar(B_CBE));
            progress = true;
          }
        }
        if constexpr (kGate) {
          // z(k) into the X̃ blocks once S_c(k) is done with them
          if (zc.live() && zc.k < kC && mbar_test_wait(bar(B_XTEMPTY), zc.k & 1u)) {
            mbar_arrive_expect_tx(bar(B_ZF), L::kHeads * kBlk);
            tma_load_3d(sbase + L::kOffXt, &tm_z, bar(B_ZF), zc.w.h[0] * kP, zc.c * kQ, zc.w.b);
            if (L::kHeads == 2)
              tma_load_3d(sbase + L::kOffXt + kBlk, &tm_z, bar(B_ZF), zc.w.h[1] * kP, zc.c * kQ, zc.w.b);
            zc.next(p);
            progress = true;
          }
        }
        if (progress) {
          t_idle = globaltimer_ns();
        } else if (*ctl.abort) {
          ok = false;
        } else if (globaltimer_ns() - t_idle > ctl.timeout) {
          raise_abort(ctl);
          ok = false;
        } else {
          __nanosleep(32);  // leave the issue slots to the warps doing the work
        }
      }
      if constexpr (kGate) {
        // a z load still in flight lands before the CTA exits
        if (!ok && zc.k > 0) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar(B_ZF), (zc.k - 1) & 1u) && globaltimer_ns() - t0 < 10000000ull) {
          }
        }
      }
      // wait for every MMA issued to finish before TMEM is released
      mma_commit(bar(B_DRAIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(B_DRAIN), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp == 3 && L::kHeads == 1) {
    // one head per CTA (state size 256): no second cumsum warp; this warp idles
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ chunk_cumsum
    // warp 2: head 0, warp 3: head 1
    // The Δ of the next chunk are loaded while this chunk's scalars are
    // formed (the loads are strided by H and take a full memory latency).
    const int hh = warp - 2;
    const float kLog2e = 1.4426950408889634f;
    int j = 0, c = 0;
    Unit w{};
    bool more = cta_unit(p, 0, w);
    if (more) c = w.c0;
    float dn[4], tn[4];
    // With retrieval rank R the chunk's rows are (token, rank) pairs, R rows a
    // token: every row carries its token's Δ as input weight, and only a
    // token's first row its decay (so the in-chunk sums are per token).
    const uint32_t rl2 = kRank ? (uint32_t)p.rank_log2 : 0u;
    const uint32_t rmask = (1u << rl2) - 1u;
    // Δ pre-processing: the raw dt and dt_bias are loaded here and combined
    // when the chunk is taken up, so that the loads stay in flight meanwhile
    float bn = 0.f;    // dt_bias of the loaded chunk's head
    uint32_t vn = 0u;  // bit e: row 4 lane + e of the loaded chunk is a token (< L)
    auto load_dt = [&](const Unit& wu, int cc) {
      const int head = hh ? wu.h[1] : wu.h[0];
      if constexpr (kDelta) {
        bn = p.dt_bias ? p.dt_bias[head] : 0.f;
        vn = 0u;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = cc * kQ + 4 * lane + e;
        float v = 0.f;
        if (row < p.L) {
          const int t = row >> rl2;
          v = p.dt[((int64_t)wu.b * (kRank ? p.Ltok : p.L) + t) * p.H + head];
          if constexpr (kDelta) vn |= 1u << e;
        }
        dn[e] = v;
        if constexpr (kRot) tn[e] = row < p.L ? p.theta[((int64_t)wu.b * p.L + row) * p.H + head] : 0.f;
      }
    };
    if (more) load_dt(w, c);
    uint32_t k = 0;
    bool ok = true;
    while (ok && more) {
      float d[4], th[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = dn[e];
        if constexpr (kDelta) {  // Δ = [softplus](dt + dt_bias); rows past L stay 0
          if ((vn >> e) & 1u) {
            v += bn;
            if (p.dt_softplus) v = softplus(v);
          }
        }
        d[e] = v;
        th[e] = kRot ? tn[e] : 0.f;
      }
      const float a2 = p.A[hh ? w.h[1] : w.h[0]] * kLog2e;
      // advance to the next chunk of this CTA and start its loads
      if (++c >= w.c1) {
        Unit wn;
        more = cta_unit(p, ++j, wn);
        if (more) {
          c = wn.c0;
          load_dt(wn, c);
          w = wn;
        }
      } else {
        load_dt(w, c);
      }
      {
        const uint32_t slot = k % kScalSlots, sph = (k / kScalSlots) & 1u;
        if (!(ok = wait_bar(bar(B_CSE0 + slot), sph ^ 1u, ctl))) break;
        {
          float cs[4];
          float run = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (((4u * lane + e) & rmask) == 0u) run += d[e] * a2;
            cs[e] = run;
          }
          float incl = run;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float up = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += up;
          }
          const float excl = incl - run;
          const float last = __shfl_sync(0xffffffffu, incl, 31);
          float c2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) c2[e] = excl + cs[e];
          // reference of each row quarter: cs at rows 0, 32, 64, 96 (lanes 0, 8, 16, 24, element 0)
          const float r0 = __shfl_sync(0xffffffffu, c2[0], 0);
          const float r1 = __shfl_sync(0xffffffffu, c2[0], 8);
          const float r2 = __shfl_sync(0xffffffffu, c2[0], 16);
          const float r3 = __shfl_sync(0xffffffffu, c2[0], 24);
          const float rq = lane < 8 ? r0 : lane < 16 ? r1 : lane < 24 ? r2 : r3;  // own quarter's reference
          float* sc = reinterpret_cast<float*>(gbase + L::kOffScal + slot * L::kScalSlotBytes + hh * L::kScalHeadBytes);
          // complex decay: the in-chunk sums φ of θ, cos φ and sin φ of every
          // row and of the chunk's last row (the rotation the chunk applies)
          float cph[4] = {1.f, 1.f, 1.f, 1.f}, sph[4] = {0.f, 0.f, 0.f, 0.f}, cL = 1.f, sL = 0.f;
          if constexpr (kRot) {
            float ps[4];
            float prun = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              prun += th[e];
              ps[e] = prun;
            }
            float pincl = prun;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const float up = __shfl_up_sync(0xffffffffu, pincl, o);
              if (lane >= o) pincl += up;
            }
            const float pexcl = pincl - prun;
            sincosf(__shfl_sync(0xffffffffu, pincl, 31), &sL, &cL);
#pragma unroll
            for (int e = 0; e < 4; ++e) sincosf(pexcl + ps[e], &sph[e], &cph[e]);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = 4 * lane + e;
            sc[SC_CS2 + i] = c2[e];
            sc[SC_U + i] = ex2(c2[e] - rq);
            sc[SC_EJ + i] = d[e] > 0.f ? __log2f(d[e]) - c2[e] : -INFINITY;
            const float wv = ex2(last - c2[e]) * d[e];
            if constexpr (kRot) {
              sc[SC_ECS + i] = ex2(c2[e]);
              const float v1 = ex2(r1 - c2[e]) * d[e], v2 = ex2(r2 - c2[e]) * d[e], v3 = ex2(r3 - c2[e]) * d[e];
              // Re / Im weights of X̃: Δ_j e^{cs_last − cs_j} (cos, sin)(φ_last − φ_j);
              // the mask's column factors v_q[j] (cos φ_j, sin φ_j)
              const float wr = wv * fmaf(cL, cph[e], sL * sph[e]);
              const float wi = wv * fmaf(sL, cph[e], -cL * sph[e]);
              reinterpret_cast<uint32_t*>(sc)[SC_W + i] = pack_bf16x2(wr, wr);
              reinterpret_cast<uint32_t*>(sc)[SC_WI + i] = pack_bf16x2(wi, wi);
              sc[SC_CPH + i] = cph[e];
              sc[SC_SPH + i] = sph[e];
              if (i < 32) sc[SC_V + i] = v1 * cph[e];
              if (i < 64) sc[SC_V + 32 + i] = v2 * cph[e];
              if (i < 96) sc[SC_V + 96 + i] = v3 * cph[e];
              if (i < 32) sc[SC_VS + i] = v1 * sph[e];
              if (i < 64) sc[SC_VS + 32 + i] = v2 * sph[e];
              if (i < 96) sc[SC_VS + 96 + i] = v3 * sph[e];
            } else {
              reinterpret_cast<uint32_t*>(sc)[SC_W + i] = pack_bf16x2(wv, wv);  // w as a bf16 pair
              sc[SC_ECS + i] = ex2(c2[e]);
              // v_q[j] = 2^(r_q − cs_j) Δ_j for the quarters q below row j's own
              if (i < 32) sc[SC_V + i] = ex2(r1 - c2[e]) * d[e];       // q = 1: j in [0, 32)
              if (i < 64) sc[SC_V + 32 + i] = ex2(r2 - c2[e]) * d[e];  // q = 2: j in [0, 64)
              if (i < 96) sc[SC_V + 96 + i] = ex2(r3 - c2[e]) * d[e];  // q = 3: j in [0, 96)
            }
          }
          if (lane == 0) {
            if constexpr (kRot) {
              sc[SC_DECAY] = ex2(last) * cL;
              sc[SC_DECAY_IM] = ex2(last) * sL;
            } else {
              sc[SC_DECAY] = ex2(last);
            }
          }
        }
        if (lane == 0) trace_ev(p.trace, k, E_CS);
        mbar_arrive(bar(B_CSF0 + slot));
      }
      ++k;
    }
  }
  } else {
    if constexpr (kBudget) setmaxnreg_inc<176>();
    // ------------------------------------------------------------ head warpgroups
    // warps 4-7: head 0, warps 8-11: head 1.  Per chunk: X̃ rows, the decay
    // mask, the state update (thread = state row n) and the y epilogue
    // (thread = token row i) of the warpgroup's head.
    const uint32_t hh = warp >= 8 ? 1u : 0u;
    const uint32_t q = warp & 3;
    const uint32_t row = 32 * q + lane;
    const uint32_t lane_addr = (32u * q) << 16;
    const int ltid = threadIdx.x - (hh ? 256 : 128);  // 0..127 within the warpgroup
    const bool rec = hh == 0;                          // head 0 records the trace
    // head (of the CTA's pair) whose mask, X̃ and y this warpgroup works on;
    // at state size 256 the CTA has one head and the two warpgroups split its
    // work (mask column blocks, X̃ rows, y columns, state rows n); with the
    // complex decay likewise, the state split by columns p instead
    constexpr bool kOne = NS == 256 || kRot;  // one head per CTA
    const uint32_t ch = kOne ? 0u : hh;
    {
      // mask slabs above the diagonal block stay zero for the whole kernel
      uint32_t z[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) z[e] = 0u;
      // (at state size 256 each warpgroup clears the slabs of its own parity,
      // so that it never overwrites a slab the other one writes)
#pragma unroll
      for (uint32_t e = 0; e < 4; ++e)
        if (e > q && (!kOne || (e & 1u) == hh)) tmem_st16(tmem + lane_addr + kTmMK + 64u * ch + 16u * e, z);
      tmem_st_wait();
    }
    uint4* xt = reinterpret_cast<uint4*>(gbase + L::kOffXt + ch * kBlk);
    // The fp32 state lives in registers.  NS = 128: thread = state row n of
    // its warpgroup's head, all 64 columns p.  NS = 256: thread = state row
    // n = 128 hh + (TMEM lane) of the one head, all 64 columns p.  NS = 64:
    // thread = row (head, p) of the pair (the TMEM lane of S_c), state
    // columns n in [32 hh, 32 hh + 32).  Complex decay: thread = state row n
    // of the one head, columns p in [32 hh, 32 hh + 32), Re parts in values
    // 0-31 and Im parts in 32-63.
    constexpr int kHS = NS == 64 ? 32 : kP;
    uint4* hb = reinterpret_cast<uint4*>(gbase + L::kOffHb + ((NS == 64 || kRot) ? 0u : hh * kBlk));
    // head of the pair whose state this thread holds
    const int sh = (NS == 128 && !kRot) ? (int)hh : kOne ? 0 : (int)(row >> 6);
    const int N = p.nstate;
    // offset of state value e of this thread within its head's [P][N] state
    // (complex decay: within the Re or Im part), or -1 (column past N)
    auto soff = [&](int e) -> int {
      if constexpr (kRot) return (32 * (int)hh + (e & 31)) * N + (int)row;
      if constexpr (NS == 128) return e * N + (int)row;
      if constexpr (NS == 256) return e * N + 128 * (int)hh + (int)row;
      const int n = 32 * (int)hh + e;
      return n < N ? (int)(row & 63u) * N + n : -1;
    };
    uint32_t k = 0, npub = 0;  // chunks done, segment hand-offs published
    bool ok = true;
    float hs[kHS];
    Unit w;
    for (int j = 0; ok && cta_unit(p, j, w); ++j) {
      const int head = ch ? w.h[1] : w.h[0];
      const bool live = ch == 0 || w.valid1;  // outputs of this head are written
      const float Dh = p.D ? p.D[head] : 0.f;
      const int shead = sh ? w.h[1] : w.h[0];
      const bool slive = sh == 0 || w.valid1;  // the state this thread holds is written
      const int64_t schain = (int64_t)w.b * p.H + shead;
      // ---- state entering the segment (complex decay: src_im the Im part)
      const float* src = nullptr;
      const float* src_im = nullptr;
      if (w.first) {
        src = p.init ? p.init + schain * kP * N : nullptr;
        if constexpr (kRot) src_im = p.init_im ? p.init_im + schain * kP * N : nullptr;
      } else {
        // (two-pass mode: this grid may start before the segment-combine
        // kernel has finished; wait for it and its stores before reading the
        // entering state it wrote)
        if (p.pdl) griddep_wait();
        // every thread acquires the flag itself (no CTA barrier that a thread
        // leaving on an error could strand)
        const uint32_t* flag = p.seg_flag + schain * p.nseg + w.pred;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_u32(flag) == 0u) {
          if (*ctl.abort) {
            ok = false;
            break;
          }
          if (globaltimer_ns() - t0 > ctl.timeout) {
            raise_abort(ctl);
            ok = false;
            break;
          }
          __nanosleep(128);
        }
        if (!ok) break;
        // (complex decay: a hand-off slot holds the Re part, then the Im part)
        src = p.seg_state + (schain * p.nseg + w.pred) * (kRot ? 2 : 1) * kP * N;
        if constexpr (kRot) src_im = src + kP * N;
      }
      if constexpr (kRot) {
#pragma unroll
        for (int e = 0; e < kHS; ++e) {
          const float* base = e >= 32 ? src_im : src;
          hs[e] = base ? base[soff(e)] : 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < kHS; ++e) {
          const int o = soff(e);
          hs[e] = (src && o >= 0) ? src[o] : 0.f;
        }
      }
      // hb holds h_in of one chunk; it is rewritten for chunk j once Y_off(j-1) is done
      auto write_hb = [&](uint32_t j) {
        if (!wait_bar(bar(B_HEMPTY), (j & 1u) ^ 1u, ctl)) return false;
        // NS = 128: row n of the head's [n][p] block; NS = 64: this thread's
        // half (16-byte chunks 4 hh .. 4 hh + 3) of row (head, p) of [(head, p)][n];
        // complex decay: this thread's column half (chunks 4 hh .. 4 hh + 3)
        // of row n of the Re block (values 0-31) and of the Im block (32-63)
#pragma unroll
        for (uint32_t c8 = 0; c8 < (uint32_t)kHS / 8; ++c8) {
          uint4 o;
          o.x = pack_bf16x2(hs[8 * c8 + 0], hs[8 * c8 + 1]);
          o.y = pack_bf16x2(hs[8 * c8 + 2], hs[8 * c8 + 3]);
          o.z = pack_bf16x2(hs[8 * c8 + 4], hs[8 * c8 + 5]);
          o.w = pack_bf16x2(hs[8 * c8 + 6], hs[8 * c8 + 7]);
          if constexpr (kRot)
            hb[((c8 >= 4 ? kBlk : 0u) + sw128_offset(row, 4u * hh + (c8 & 3u))) >> 4] = o;
          else
            hb[sw128_offset(row, NS == 64 ? 4u * hh + c8 : c8) >> 4] = o;
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(B_HFULL));
        return true;
      };
      if (w.c1 > w.c0 && !(ok = write_hb(k))) break;
      for (int c = w.c0; c < w.c1; ++c, ++k) {
        const uint32_t cp = k & 1u, slot = k % kScalSlots;
        const uint32_t xs = k % kXStages, xph = (k / kXStages) & 1u;
        if (!(ok = wait_bar(bar(B_CSF0 + slot), (k / kScalSlots) & 1u, ctl))) break;
        const float* sc =
            reinterpret_cast<const float*>(gbase + L::kOffScal + slot * L::kScalSlotBytes + ch * L::kScalHeadBytes);
        // ---- X̃ = w ⊙ X of this head, same swizzled layout as X.  Rows are
        // spread against the mask work, which grows with q: warp q=0 takes rows
        // 0-63, q=1 rows 64-95, q=2 rows 96-127, q=3 none (at state size 256,
        // warps q = 0, 1 of warpgroup hh take rows 64 hh + 32 q .. + 31).
        if (!(ok = wait_bar(bar(B_XF00 + 2 * ch + xs), xph, ctl))) break;
        if (!(ok = wait_bar(bar(B_XTEMPTY), cp ^ 1u, ctl))) break;
        if constexpr (kGate) {
          // the rows this warp writes may belong to another warp's z(k-1)
          if (k > 0 && !(ok = wait_bar(bar(B_ZE0 + hh), cp ^ 1u, ctl))) break;
          if (NS == 256 && k > 0 && !(ok = wait_bar(bar(B_ZE0 + (hh ^ 1u)), cp ^ 1u, ctl))) break;
        }
        if (rec && warp == 4 && lane == 0) trace_ev(p.trace, k, E_XT_START);
        {
          const uint4* xsrc = reinterpret_cast<const uint4*>(gbase + x_tile<NS>(ch, k));
          const uint32_t nrows = kOne ? (q < 2 ? 1u : 0u) : (q == 0 ? 2u : (q == 3 ? 0u : 1u));
          for (uint32_t rr = 0; rr < nrows; ++rr) {
            const uint32_t xr = kOne ? 64u * hh + 32u * q + lane
                                     : (q == 0 ? 32u * rr + lane : 32u * (q + 1) + lane);
            const uint32_t wx = reinterpret_cast<const uint32_t*>(sc)[SC_W + xr];  // (w, w) bf16
            uint4 v[8];
#pragma unroll
            for (uint32_t ch = 0; ch < 8; ++ch) v[ch] = xsrc[sw128_offset(xr, ch) >> 4];
#pragma unroll
            for (uint32_t ch = 0; ch < 8; ++ch) {
              uint4 o;
              o.x = mul_bf16x2(v[ch].x, wx);
              o.y = mul_bf16x2(v[ch].y, wx);
              o.z = mul_bf16x2(v[ch].z, wx);
              o.w = mul_bf16x2(v[ch].w, wx);
              xt[sw128_offset(xr, ch) >> 4] = o;
            }
            if constexpr (kRot) {
              // the Im weighting into the second X̃ block
              const uint32_t wi = reinterpret_cast<const uint32_t*>(sc)[SC_WI + xr];
#pragma unroll
              for (uint32_t ch = 0; ch < 8; ++ch) {
                uint4 o;
                o.x = mul_bf16x2(v[ch].x, wi);
                o.y = mul_bf16x2(v[ch].y, wi);
                o.z = mul_bf16x2(v[ch].z, wi);
                o.w = mul_bf16x2(v[ch].w, wi);
                xt[(kBlk + sw128_offset(xr, ch)) >> 4] = o;
              }
            }
          }
        }
        fence_proxy_async_smem();
        if (rec && warp == 4 && lane == 0) trace_ev(p.trace, k, E_XT_END);
        mbar_arrive(bar(B_XTFULL));
        // ---- decay mask of this head from S = C Bᵀ
        if (!(ok = wait_bar(bar(B_SFULL), cp, ctl))) break;
        if (!(ok = wait_bar(bar(B_MEMPTY), cp ^ 1u, ctl))) break;
        if (rec && warp == 7 && lane == 0) trace_ev(p.trace, k, E_MK3_START);
        tc_fence_after();
        {
          const uint32_t tS = tmem + lane_addr + kTmS;
          const uint32_t tM = tmem + lane_addr + kTmMK + 64u * ch;
          const float u_i = sc[SC_U + row];
          const float c2_i = sc[SC_CS2 + row];
          const float4* vq = reinterpret_cast<const float4*>(sc + SC_V + (q == 1 ? 0 : q == 2 ? 32 : 96));
          const float4* ejq = reinterpret_cast<const float4*>(sc + SC_EJ + 32 * q);
          // the diagonal block keeps the columns up to the last row of this
          // row's token (rows of one token all see each other's writes)
          const uint32_t rl2 = kRank ? (uint32_t)p.rank_log2 : 0u;
          const int lim = (int)((((uint32_t)lane >> rl2) + 1u) << rl2);
          // slabs kb = 0..q: left of the diagonal S · u_i · v_j, the diagonal
          // block S · 2^(cs_i − cs_j) Δ_j for j ≤ i plus D on the diagonal (the
          // skip term D x_i).  TMEM loads run one slab ahead.  At state size
          // 256 the two warpgroups share the one head's slabs: even kb to
          // warpgroup 0, odd kb to warpgroup 1.
          constexpr uint32_t kbs = kOne ? 2u : 1u;
          const uint32_t kb0 = kOne ? hh : 0u;
          // complex decay: every entry also takes cos(φ_i − φ_j) = cos φ_i cos φ_j
          // + sin φ_i sin φ_j (row factors here, column factors from the scalars)
          const float cph_i = kRot ? sc[SC_CPH + row] : 1.f, sph_i = kRot ? sc[SC_SPH + row] : 0.f;
          const float4* vsq = reinterpret_cast<const float4*>(sc + SC_VS + (q == 1 ? 0 : q == 2 ? 32 : 96));
          const float4* cpq = reinterpret_cast<const float4*>(sc + SC_CPH + 32 * q);
          const float4* spq = reinterpret_cast<const float4*>(sc + SC_SPH + 32 * q);
          uint32_t ra[32], rb[32];
          if (kb0 <= q) tmem_ld32(tS + 32u * kb0, ra);
          for (uint32_t kb = kb0; kb <= q; kb += kbs) {
            tmem_ld_wait();
            reg_fence(ra);
#pragma unroll
            for (int e = 0; e < 32; ++e) rb[e] = ra[e];
            if (kb + kbs <= q) tmem_ld32(tS + 32u * (kb + kbs), ra);
            uint32_t m[16];
            if (kRot && kb < q) {
              // S · (u_i cos φ_i · v_j cos φ_j + u_i sin φ_i · v_j sin φ_j)
              const float uc = u_i * cph_i, us = u_i * sph_i;
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                const float4 vc = vq[(32 * kb + e) >> 2];
                const float4 vs = vsq[(32 * kb + e) >> 2];
                const float a0 = __uint_as_float(rb[e]) * fmaf(uc, vc.x, us * vs.x);
                const float a1 = __uint_as_float(rb[e + 1]) * fmaf(uc, vc.y, us * vs.y);
                const float a2 = __uint_as_float(rb[e + 2]) * fmaf(uc, vc.z, us * vs.z);
                const float a3 = __uint_as_float(rb[e + 3]) * fmaf(uc, vc.w, us * vs.w);
                m[e >> 1] = pack_bf16x2(a0, a1);
                m[(e >> 1) + 1] = pack_bf16x2(a2, a3);
              }
            } else if (kb < q) {
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                const float4 v = vq[(32 * kb + e) >> 2];
                const float a0 = __uint_as_float(rb[e]) * u_i * v.x;
                const float a1 = __uint_as_float(rb[e + 1]) * u_i * v.y;
                const float a2 = __uint_as_float(rb[e + 2]) * u_i * v.z;
                const float a3 = __uint_as_float(rb[e + 3]) * u_i * v.w;
                m[e >> 1] = pack_bf16x2(a0, a1);
                m[(e >> 1) + 1] = pack_bf16x2(a2, a3);
              }
            } else if (kRot) {
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                const float4 ev = ejq[e >> 2];
                const float4 cj = cpq[e >> 2];
                const float4 sj = spq[e >> 2];
                float a0 = __uint_as_float(rb[e]) * ex2(c2_i + ev.x) * fmaf(cph_i, cj.x, sph_i * sj.x);
                float a1 = __uint_as_float(rb[e + 1]) * ex2(c2_i + ev.y) * fmaf(cph_i, cj.y, sph_i * sj.y);
                float a2 = __uint_as_float(rb[e + 2]) * ex2(c2_i + ev.z) * fmaf(cph_i, cj.z, sph_i * sj.z);
                float a3 = __uint_as_float(rb[e + 3]) * ex2(c2_i + ev.w) * fmaf(cph_i, cj.w, sph_i * sj.w);
                if (e > lane) a0 = 0.f;
                if (e + 1 > lane) a1 = 0.f;
                if (e + 2 > lane) a2 = 0.f;
                if (e + 3 > lane) a3 = 0.f;
                if (e == lane) a0 += Dh;
                if (e + 1 == lane) a1 += Dh;
                if (e + 2 == lane) a2 += Dh;
                if (e + 3 == lane) a3 += Dh;
                m[e >> 1] = pack_bf16x2(a0, a1);
                m[(e >> 1) + 1] = pack_bf16x2(a2, a3);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                const float4 ev = ejq[e >> 2];
                float a0 = __uint_as_float(rb[e]) * ex2(c2_i + ev.x);
                float a1 = __uint_as_float(rb[e + 1]) * ex2(c2_i + ev.y);
                float a2 = __uint_as_float(rb[e + 2]) * ex2(c2_i + ev.z);
                float a3 = __uint_as_float(rb[e + 3]) * ex2(c2_i + ev.w);
                if (e >= lim) a0 = 0.f;
                if (e + 1 >= lim) a1 = 0.f;
                if (e + 2 >= lim) a2 = 0.f;
                if (e + 3 >= lim) a3 = 0.f;
                if (e == lane) a0 += Dh;
                if (e + 1 == lane) a1 += Dh;
                if (e + 2 == lane) a2 += Dh;
                if (e + 3 == lane) a3 += Dh;
                m[e >> 1] = pack_bf16x2(a0, a1);
                m[(e >> 1) + 1] = pack_bf16x2(a2, a3);
              }
            }
            tmem_st16(tM + 16u * kb, m);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        if (rec && warp == 7 && lane == 0) trace_ev(p.trace, k, E_MK3_END);
        if (rec && warp == 4 && lane == 0) trace_ev(p.trace, k, E_MK0_END);
        mbar_arrive(bar(B_MFULL0 + hh));
        // ---- state_passing: h_in[k+1] = decay h_in[k] + S_c
        const float* scs =
            reinterpret_cast<const float*>(gbase + L::kOffScal + slot * L::kScalSlotBytes + (uint32_t)sh * L::kScalHeadBytes);
        const float decay = scs[SC_DECAY];  // complex decay: its Re part, scs[SC_DECAY_IM] the Im part
        const float ecs_i = sc[SC_ECS + row];
        if (!(ok = wait_bar(bar(B_SCFULL), cp, ctl))) break;
        if (rec && ltid == 0) trace_ev(p.trace, k, E_ST_START);
        tc_fence_after();
        if constexpr (kRot) {
          // S_cᵀ: TMEM lane = state row n, columns p of Re (0-63) then Im (64-127);
          // this warpgroup's columns 32 hh .. 32 hh + 31 of both.
          // h ← (d_re + i d_im) h + S_c
          const float dim = scs[SC_DECAY_IM];
          uint32_t r0[32], r1[32];
          tmem_ld32(tmem + lane_addr + kTmSc + 32u * hh, r0);
          tmem_ld32(tmem + lane_addr + kTmSc + 64u + 32u * hh, r1);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          tc_fence_before();
          mbar_arrive(bar(B_SCEMPTY));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float re = hs[e], im = hs[32 + e];
            hs[e] = fmaf(decay, re, fmaf(-dim, im, __uint_as_float(r0[e])));
            hs[32 + e] = fmaf(dim, re, fmaf(decay, im, __uint_as_float(r1[e])));
          }
        } else if constexpr (NS != 64) {
          // S_cᵀ: TMEM lane = state row n (of head hh, or of n half hh at state size 256), column = p
          uint32_t r0[32], r1[32];
          tmem_ld32(tmem + lane_addr + kTmSc + 64u * hh, r0);
          tmem_ld32(tmem + lane_addr + kTmSc + 64u * hh + 32u, r1);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          tc_fence_before();
          mbar_arrive(bar(B_SCEMPTY));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            hs[e] = fmaf(decay, hs[e], __uint_as_float(r0[e]));
            hs[32 + e] = fmaf(decay, hs[32 + e], __uint_as_float(r1[e]));
          }
        } else {
          // S_c: TMEM lane = (head, p) of the pair, column = n
          uint32_t r0[32];
          tmem_ld32(tmem + lane_addr + kTmSc + 32u * hh, r0);
          tmem_ld_wait();
          reg_fence(r0);
          tc_fence_before();
          mbar_arrive(bar(B_SCEMPTY));
#pragma unroll
          for (int e = 0; e < 32; ++e) hs[e] = fmaf(decay, hs[e], __uint_as_float(r0[e]));
        }
        if (c + 1 < w.c1 && !(ok = write_hb(k + 1))) break;
        if (rec && ltid == 0) trace_ev(p.trace, k, E_ST_END);
        // ---- y epilogue: y_i = Y_i + 2^cs_i Y_off,i, staged into the X tile
        if (!(ok = wait_bar(bar(B_YFULL), cp, ctl))) break;
        if (!(ok = wait_bar(bar(B_YOFFFULL), cp, ctl))) break;
        if constexpr (kGate) {
          if (!(ok = wait_bar(bar(B_ZF), cp, ctl))) break;
        }
        if (rec && ltid == 0) trace_ev(p.trace, k, E_Y_START);
        tc_fence_after();
        {
          uint4* yt = reinterpret_cast<uint4*>(gbase + x_tile<NS>(ch, k));
          const uint4* zt = reinterpret_cast<const uint4*>(gbase + L::kOffXt + ch * kBlk);  // z tile (gate)
          const uint32_t tY = tmem + lane_addr + kTmSc + 64u * ch;
          const uint32_t tO = tmem + lane_addr + kTmYoff + 64u * ch;
          if constexpr (kRot) {
            // y_i = Y_i + 2^cs_i (cos φ_i Y_off,Re − sin φ_i Y_off,Im), columns
            // 32 hh .. 32 hh + 31 in two slices of 16 (Y_off Re in columns 0-63,
            // Im in 64-127)
            const float ec = ecs_i * sc[SC_CPH + row], es = -ecs_i * sc[SC_SPH + row];
#pragma unroll
            for (uint32_t sl = 0; sl < 2; ++sl) {
              uint32_t ya[16], oa[16], ob[16];
              const uint32_t col = 32u * hh + 16u * sl;
              tmem_ld16(tY + col, ya);
              tmem_ld16(tO + col, oa);
              tmem_ld16(tO + 64u + col, ob);
              tmem_ld_wait();
              reg_fence16(ya);
              reg_fence16(oa);
              reg_fence16(ob);
              if (sl == 1) {
                tc_fence_before();
                mbar_arrive(bar(B_SYEMPTY));
              }
#pragma unroll
              for (uint32_t cq = 0; cq < 2; ++cq) {
                uint32_t vw[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                  const int e = 8 * cq + 2 * e2;
                  const float y0 = fmaf(ec, __uint_as_float(oa[e]),
                                        fmaf(es, __uint_as_float(ob[e]), __uint_as_float(ya[e])));
                  const float y1 = fmaf(ec, __uint_as_float(oa[e + 1]),
                                        fmaf(es, __uint_as_float(ob[e + 1]), __uint_as_float(ya[e + 1])));
                  vw[e2] = pack_bf16x2(y0, y1);
                }
                yt[sw128_offset(row, 4 * hh + 2 * sl + cq) >> 4] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
              }
            }
          }
          // columns p in halves of 32: both halves, or at state size 256 half hh
          constexpr uint32_t kHalves = kRot ? 0u : NS == 256 ? 1u : 2u;
#pragma unroll
          for (uint32_t hi = 0; hi < kHalves; ++hi) {
            const uint32_t half = NS == 256 ? hh : hi;
            uint32_t ya[32], oa[32];
            tmem_ld32(tY + 32u * half, ya);
            tmem_ld32(tO + 32u * half, oa);
            tmem_ld_wait();
            reg_fence(ya);
            reg_fence(oa);
            if (hi == kHalves - 1) {
              tc_fence_before();
              mbar_arrive(bar(B_SYEMPTY));
            }
#pragma unroll
            for (uint32_t cq = 0; cq < 4; ++cq) {
              uint32_t vw[4], zw[4] = {0u, 0u, 0u, 0u};
              if constexpr (kGate) {
                const uint4 zz = zt[sw128_offset(row, 4 * half + cq) >> 4];
                zw[0] = zz.x;
                zw[1] = zz.y;
                zw[2] = zz.z;
                zw[3] = zz.w;
              }
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2) {
                const int e = 8 * cq + 2 * e2;  // column within the half
                float y0 = fmaf(ecs_i, __uint_as_float(oa[e]), __uint_as_float(ya[e]));
                float y1 = fmaf(ecs_i, __uint_as_float(oa[e + 1]), __uint_as_float(ya[e + 1]));
                if constexpr (kGate) {  // y · silu(z)
                  y0 *= silu(bf16lo_to_f(zw[e2]));
                  y1 *= silu(bf16hi_to_f(zw[e2]));
                }
                vw[e2] = pack_bf16x2(y0, y1);
              }
              yt[sw128_offset(row, 4 * half + cq) >> 4] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
            }
          }
        }
        fence_proxy_async_smem();
        if (rec && ltid == 0) trace_ev(p.trace, k, E_Y_END);
        mbar_arrive(bar(B_YST00 + 2 * hh + xs));
        mbar_arrive(bar(B_CSE0 + slot));
        if constexpr (kGate) mbar_arrive(bar(B_ZE0 + hh));
      }
      if (!ok) break;
      // ---- publish the state leaving the segment
      if (slive) {
        float* dst = nullptr;
        float* dst_im = nullptr;  // complex decay: the Im part
        if (w.last) {
          dst = p.final_state ? p.final_state + schain * kP * N : nullptr;
          if constexpr (kRot) dst_im = p.final_im ? p.final_im + schain * kP * N : nullptr;
        } else if (p.publish) {
          dst = p.seg_state + (schain * p.nseg + w.pub) * (kRot ? 2 : 1) * kP * N;
          if constexpr (kRot) dst_im = dst + kP * N;
        }
        if constexpr (kRot) {
#pragma unroll
          for (int e = 0; e < kHS; ++e) {
            float* d = e >= 32 ? dst_im : dst;
            if (d) d[soff(e)] = hs[e];
          }
        } else if (dst) {
#pragma unroll
          for (int e = 0; e < kHS; ++e) {
            const int o = soff(e);
            if (o >= 0) dst[o] = hs[e];
          }
        }
      }
      if (p.publish && !w.last) {
        // Lane 3 of the producer warp raises the flag once all 128 threads
        // have stored their rows and arrived (the arrive releases the stores
        // at CTA scope, the flag store at GPU scope), so no thread here waits
        // for its stores to drain.  Hand-off n+1 waits until hand-off n has
        // been taken.
        if (npub > 0 && !(ok = wait_bar(bar(B_PUBACK), (npub - 1) & 1u, ctl))) break;
        mbar_arrive(bar(B_PUB0 + hh));
        ++npub;
      }
    }
  }

  __syncthreads();
  if (p.trace != nullptr && threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas) {
    long long* t = const_cast<long long*>(p.trace) + kTraceChunks * kTraceEvents + 6 * blockIdx.x;
    t[1] = (long long)globaltimer_ns();
    t[5] = clock64();
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    t[3] = smid;
    Unit w;
    long long n = 0;
    for (int j = 0; cta_unit(p, j, w); ++j) n += w.c1 - w.c0;
    t[2] = n;
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmCols);
  }
}

// ---------------------------------------------------------------- segment states (two-pass mode)
// When there are fewer sequences than SMs, a sequence's segments cannot wait
// for one another without leaving SMs idle.  The forward pass then runs in
// two passes: ssd_states_kernel computes, for every segment, the state its
// chunks produce from a zero entering state and the product of the chunk
// decays (the recurrence of §2.1.2 lifted to segments, as the chunk states
// are lifted to chunks); ssd_seg_combine_kernel chains the segments
// (h_in[s+1] = D_s · h_in[s] + h_loc[s]) and publishes every entering state;
// the fused kernel then runs all segments at once, none waiting.
//
// ssd_states_kernel: per chunk, X̃ = w ⊙ X (head warpgroups), S_cᵀ = Bᵀ X̃
// (one MMA, both heads, as in the fused kernel) and h ← decay · h + S_c.
// kMode 1 (the backward pass's recomputed states): units [0, so.units_fwd)
// are whole sequences of the forward states, started from init_state, the
// state entering each chunk written in bf16 to so.hin[b][c][h][p][n]; the
// units after them walk the adjoint states of the same sequences on
// (C, dy) (maps tm_x2, tm_b2), chunks last to first, weights 2^{cs_i}, from
// so.dfinal: the adjoint leaving each chunk goes to so.gout in bf16 (Gout[c])
// and the adjoint entering chunk 0 to so.dinit.  The adjoint recurrence is
// the state's, G ← 2^{cs_last} G + Σ_i 2^{cs_i} dy_i C_iᵀ.  Both kinds share
// one grid, so its CTAs take the two sets of sequences as they come free.
namespace st {
constexpr uint32_t kOffB = 0;                              // B ring [stage] (two 64-column blocks)
constexpr uint32_t kOffX = 2 * 2 * kBlk;                   // X ring [head][stage]
constexpr uint32_t kOffXt = kOffX + 2 * kXStages * kBlk;   // X̃ [head]
constexpr uint32_t kOffScal = kOffXt + 2 * kBlk;           // [slot][head]: w (bf16 pairs) [128], decay
constexpr uint32_t kScalHead = 132 * 4;
constexpr int kSlots = 4;
constexpr uint32_t kOffBar = kOffScal + kSlots * 2 * kScalHead;
enum : uint32_t {
  BF0 = 0, BF1, BE0, BE1,          // B ring [stage]: landed / S_c done with it
  XF00, XF01, XF10, XF11,          // X ring [head][stage]: landed
  XE00, XE01, XE10, XE11,          // X ring [head][stage]: X̃ formed from it
  CSF0, CSF1, CSF2, CSF3,          // scalar ring [slot]: written
  CSE0, CSE1, CSE2, CSE3,          // scalar ring [slot]: read by both head warpgroups
  XTFULL, XTEMPTY,                 // X̃ written / S_c done with it
  SCFULL, SCEMPTY,                 // S_c in TMEM / read
  PUB0, PUB1,                      // state walks: the state at the cut stored by head warpgroup 0 / 1
  DRAIN,
  kBars
};
constexpr uint32_t kOffMisc = kOffBar + kBars * 8;
constexpr uint32_t kSmemAlloc = kOffMisc + 16 + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");
constexpr uint32_t kTmCols = 128;
}  // namespace st

struct SeqOut {
  __nv_bfloat16* hin;    // [B][nc][H][P][N]: the state entering each chunk
  __nv_bfloat16* gout;   // [B][nc][H][P][N]: the adjoint leaving each chunk
  const float* dfinal;   // [B][H][P][N] or null: the adjoint leaving the last chunk
  float* dinit;          // [B][H][P][N] or null: the adjoint entering chunk 0
  int32_t units_fwd;     // walks (head-pair sequences) before the adjoint ones
  uint32_t* flag;        // [walk][2]: 1 once the state handed over at the walk's cut is stored
  float* slot;           // [walk][2][P][N]: that state, fp32
};

// kMode 1: the j-th piece of walk this CTA owns, in processing order (false
// past the last).  The 2 · units_fwd walks of nc steps, laid end to end, are
// cut into gridDim.x equal ranges (at least one walk long), as cta_unit cuts
// the fused kernel's sequences: last walk first, so a CTA hands a state over
// at most once in each direction and never waits on a later piece of its
// own.  w.c0, w.c1 are steps (the adjoint's step j is chunk nc − 1 − j);
// w.pub is the walk index.
__device__ __forceinline__ bool walk_piece(const FusedParams& p, const SeqOut& so, int j, Unit& w, bool& adj) {
  const int64_t total = (int64_t)2 * so.units_fwd * p.nc;
  const int64_t s = (int64_t)blockIdx.x * total / gridDim.x;
  const int64_t e = (int64_t)(blockIdx.x + 1) * total / gridDim.x;
  const int64_t x = (e - 1) / p.nc - j;
  if (e <= s || x < s / p.nc) return false;
  adj = x >= so.units_fwd;
  chain_info(p, (int)(adj ? x - so.units_fwd : x), w);
  const int64_t base = x * p.nc;
  w.c0 = (int)((s > base ? s : base) - base);
  w.c1 = (int)((e < base + p.nc ? e : base + p.nc) - base);
  w.first = w.c0 == 0;
  w.last = w.c1 == p.nc;
  w.s = 0;
  w.pred = 0;
  w.pub = (int)x;
  return true;
}

template <bool kDelta, int kMode = 0>
__global__ void __launch_bounds__(384, 1)
    ssd_states_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_x2, const __grid_constant__ CUtensorMap tm_b2,
                      const FusedParams p, float* seg_local, float* seg_decay, const SeqOut so) {
  constexpr bool kHin = kMode != 0;
  // the jj-th unit of this CTA: a segment (round-robin), or a piece of a
  // forward or adjoint walk (kMode 1, contiguous ranges)
  auto next_unit = [&](int jj, Unit& w, bool& adj) -> bool {
    if constexpr (kHin) {
      return walk_piece(p, so, jj, w, adj);
    } else {
      const int u = (int)blockIdx.x + jj * (int)gridDim.x;
      if (u >= p.units) return false;
      adj = false;
      w = unit_info(p, u);
      return true;
    }
  };
  // chunk of step j of a unit (the adjoint walks its chunks last to first)
  auto chunk_of = [&](const Unit& w, int j, bool adj) { return adj ? p.nc - 1 - (w.c0 + j) : w.c0 + j; };
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (sbase - raw);
  auto bar = [&](uint32_t i) { return sbase + st::kOffBar + 8u * i; };
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(gbase + st::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(gbase + st::kOffMisc + 4);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  auto xtile = [&](uint32_t hh, uint32_t k) { return st::kOffX + (hh * kXStages + (k % kXStages)) * kBlk; };
  // the workspace's status word and flags start at zero on every call (read
  // by the later kernels of the call only, which start after this one ends)
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < p.zero_words; i += gridDim.x * blockDim.x)
    reinterpret_cast<uint4*>(p.err)[i] = make_uint4(0u, 0u, 0u, 0u);

  if (threadIdx.x == 0) {
    uint32_t counts[st::kBars];
    for (uint32_t i = 0; i < st::kBars; ++i) counts[i] = 1;  // TMA expect_tx, MMA commits
    counts[st::XE00] = counts[st::XE01] = counts[st::XE10] = counts[st::XE11] = 128;  // the head's warpgroup
    for (int i = 0; i < st::kSlots; ++i) {
      counts[st::CSF0 + i] = 64;   // both cumsum warps
      counts[st::CSE0 + i] = 256;  // both head warpgroups
    }
    counts[st::XTFULL] = counts[st::SCEMPTY] = 256;
    counts[st::PUB0] = counts[st::PUB1] = 128;  // one head warpgroup each
    for (uint32_t i = 0; i < st::kBars; ++i) mbar_init(bar(i), counts[i]);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + st::kOffMisc, st::kTmCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_b);
    if constexpr (kHin) {
      tma_prefetch_desc(&tm_x2);
      tma_prefetch_desc(&tm_b2);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (kHin && lane == 3) {
      // ---- hand-off flags (kMode 1): once both head warpgroups have stored
      // the state at this CTA's cut, make the stores visible at GPU scope and
      // raise the two heads' flags
      Unit w;
      bool adj;
      uint32_t npub = 0;
      for (int jj = 0; next_unit(jj, w, adj); ++jj) {
        if (w.last) continue;
        if (!wait_bar(bar(st::PUB0), npub & 1u, ctl) || !wait_bar(bar(st::PUB1), npub & 1u, ctl)) break;
        __threadfence();
        st_release_u32(so.flag + 2 * w.pub, 1u);
        st_release_u32(so.flag + 2 * w.pub + 1, 1u);
        ++npub;
      }
    }
    // ---- producers: lane 0 the B tiles (2-stage ring), lanes 1, 2 the X tiles of head 0 / 1
    if (lane < 3) {
      uint32_t k = 0;
      bool ok = true;
      Unit w;
      bool adj;
      for (int jj = 0; ok && next_unit(jj, w, adj); ++jj) {
        for (int j = 0; j < w.c1 - w.c0; ++j, ++k) {
          const int c = chunk_of(w, j, adj);
          const uint32_t s = k % 2u, ph = (k / 2u) & 1u;
          const CUtensorMap* mx = adj ? &tm_x2 : &tm_x;  // (the adjoint: dy, C)
          const CUtensorMap* mb = adj ? &tm_b2 : &tm_b;
          if (lane == 0) {
            if (!(ok = wait_bar(bar(st::BE0 + s), ph ^ 1u, ctl))) break;
            mbar_arrive_expect_tx(bar(st::BF0 + s), 2 * kBlk);
            tma_load_3d(sbase + st::kOffB + s * 2 * kBlk, mb, bar(st::BF0 + s), w.g * kN, c * kQ, w.b);
            tma_load_3d(sbase + st::kOffB + s * 2 * kBlk + kBlk, mb, bar(st::BF0 + s), w.g * kN + 64, c * kQ, w.b);
          } else {
            const uint32_t hh = lane - 1, xs = k % kXStages, xph = (k / kXStages) & 1u;
            if (!(ok = wait_bar(bar(st::XE00 + 2 * hh + xs), xph ^ 1u, ctl))) break;
            mbar_arrive_expect_tx(bar(st::XF00 + 2 * hh + xs), kBlk);
            tma_load_3d(sbase + xtile(hh, k), mx, bar(st::XF00 + 2 * hh + xs), (hh ? w.h[1] : w.h[0]) * kP, c * kQ,
                        w.b);
          }
        }
      }
      if (!ok) {
        // let the loads already issued land before the CTA exits
        for (uint32_t j = (k >= 2 ? k - 2 : 0); j < k; ++j) {
          const uint32_t b2 = lane == 0 ? bar(st::BF0 + j % 2u) : bar(st::XF00 + 2 * (lane - 1) + j % kXStages);
          const uint32_t par = lane == 0 ? ((j / 2u) & 1u) : ((j / kXStages) & 1u);
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(b2, par) && globaltimer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA: S_cᵀ(k) = Bᵀ [X̃_0 | X̃_1], one stream
    if (lane == 0) {
      const uint64_t dBm = smem_desc_sw128(sbase + st::kOffB, kBlk, 1024);
      const uint64_t dXt = smem_desc_sw128(sbase + st::kOffXt, kBlk, 1024);
      uint32_t k = 0;
      bool ok = true;
      Unit w;
      bool adj;
      for (int jj = 0; ok && next_unit(jj, w, adj); ++jj) {
        for (int j = 0; j < w.c1 - w.c0; ++j, ++k) {
          const uint32_t s = k % 2u;
          if (!(ok = wait_bar(bar(st::BF0 + s), (k / 2u) & 1u, ctl) && wait_bar(bar(st::XTFULL), k & 1u, ctl) &&
                     wait_bar(bar(st::SCEMPTY), (k & 1u) ^ 1u, ctl)))
            break;
          tc_fence_after();
          mma_k128_ss<KSTEP_ROWS, KSTEP_ROWS>(tmem, dBm + (uint64_t)(s * ((2 * kBlk) >> 4)), dXt, kIdescSc);
          mma_commit(bar(st::SCFULL));
          mma_commit(bar(st::XTEMPTY));
          mma_commit(bar(st::BE0 + s));
        }
      }
      mma_commit(bar(st::DRAIN));
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar(st::DRAIN), 0) && globaltimer_ns() - t0 < 100000000ull) {
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ---- per-chunk w and decay of one head (warp 2: head 0, warp 3: head 1)
    const int hh = warp - 2;
    const float kLog2e = 1.4426950408889634f;
    uint32_t k = 0;
    bool ok = true;
    Unit w;
    bool adj;
    for (int jj = 0; ok && next_unit(jj, w, adj); ++jj) {
      const int head = hh ? w.h[1] : w.h[0];
      const float a2 = p.A[head] * kLog2e;
      for (int j = 0; j < w.c1 - w.c0; ++j, ++k) {
        const int c = chunk_of(w, j, adj);
        float d[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = c * kQ + 4 * lane + e;
          float v = 0.f;
          if (t < p.L) {
            v = p.dt[((int64_t)w.b * p.L + t) * p.H + head];
            if constexpr (kDelta) {
              if (p.dt_bias) v += p.dt_bias[head];
              if (p.dt_softplus) v = softplus(v);
            }
          }
          d[e] = v;
        }
        const uint32_t slot = k % st::kSlots;
        if (!(ok = wait_bar(bar(st::CSE0 + slot), ((k / st::kSlots) & 1u) ^ 1u, ctl))) break;
        float cs[4];
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          run += d[e] * a2;
          cs[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float up = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += up;
        }
        const float excl = incl - run;
        const float last = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t* sc = reinterpret_cast<uint32_t*>(gbase + st::kOffScal + (slot * 2 + hh) * st::kScalHead);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // w_i = 2^{cs_last − cs_i} Δ_i (the state), 2^{cs_i} (the adjoint; cs inclusive)
          const float wv = adj ? ex2(excl + cs[e]) : ex2(last - (excl + cs[e])) * d[e];
          sc[4 * lane + e] = pack_bf16x2(wv, wv);  // w as a bf16 pair
        }
        if (lane == 0) reinterpret_cast<float*>(sc)[128] = ex2(last);
        mbar_arrive(bar(st::CSF0 + slot));
      }
    }
  } else {
    // ---- head warpgroups (warps 4-7: head 0, 8-11: head 1): X̃ rows, the
    // state update (thread = state row n), the segment's local state
    const uint32_t hh = warp >= 8 ? 1u : 0u;
    const uint32_t q = warp & 3;
    const uint32_t row = 32 * q + lane;
    const uint32_t lane_addr = (32u * q) << 16;
    const int ltid = threadIdx.x - (hh ? 256 : 128);
    uint4* xt = reinterpret_cast<uint4*>(gbase + st::kOffXt + hh * kBlk);
    uint32_t k = 0;
    bool ok = true;
    float hs[kP];
    Unit w;
    bool adj;
    for (int jj = 0; ok && next_unit(jj, w, adj); ++jj) {
      const int head = hh ? w.h[1] : w.h[0];
      const bool live = hh == 0 || w.valid1;
      const int64_t hchain = (int64_t)w.b * p.H + head;
      {
        // the segment starts from zero; a walk from init_state (the adjoint:
        // from dfinal), or, for a piece after the cut, from the state its
        // predecessor handed over
        const float* start = !kHin ? nullptr : adj ? so.dfinal : p.init;
        if (kHin && !w.first) {
          const uint32_t* flag = so.flag + 2 * w.pub + hh;
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_u32(flag) == 0u) {
            if (*ctl.abort) {
              ok = false;
              break;
            }
            if (globaltimer_ns() - t0 > ctl.timeout) {
              raise_abort(ctl);
              ok = false;
              break;
            }
            __nanosleep(64);
          }
          if (!ok) break;
          start = so.slot + (int64_t)(2 * w.pub + hh) * kP * kN;
        }
        const float* src = start ? start + ((kHin && !w.first) ? 0 : hchain * kP * kN) : nullptr;
#pragma unroll
        for (int pp = 0; pp < kP; ++pp) hs[pp] = src ? src[pp * kN + row] : 0.f;
      }
      float dprod = 1.f;  // product of the chunk decays of the segment
      for (int j = 0; j < w.c1 - w.c0; ++j, ++k) {
        const int c = chunk_of(w, j, adj);
        const uint32_t cp = k & 1u, slot = k % st::kSlots;
        const uint32_t xs = k % kXStages, xph = (k / kXStages) & 1u;
        if (!(ok = wait_bar(bar(st::CSF0 + slot), (k / st::kSlots) & 1u, ctl))) break;
        const uint32_t* sc = reinterpret_cast<const uint32_t*>(gbase + st::kOffScal + (slot * 2 + hh) * st::kScalHead);
        // X̃ = w ⊙ X, same swizzled layout as X; each warp takes 32 rows
        if (!(ok = wait_bar(bar(st::XF00 + 2 * hh + xs), xph, ctl))) break;
        if (!(ok = wait_bar(bar(st::XTEMPTY), cp ^ 1u, ctl))) break;
        {
          const uint4* xsrc = reinterpret_cast<const uint4*>(gbase + xtile(hh, k));
          const uint32_t xr = row;
          const uint32_t wx = sc[xr];
          uint4 v[8];
#pragma unroll
          for (uint32_t ch = 0; ch < 8; ++ch) v[ch] = xsrc[sw128_offset(xr, ch) >> 4];
#pragma unroll
          for (uint32_t ch = 0; ch < 8; ++ch) {
            uint4 o;
            o.x = mul_bf16x2(v[ch].x, wx);
            o.y = mul_bf16x2(v[ch].y, wx);
            o.z = mul_bf16x2(v[ch].z, wx);
            o.w = mul_bf16x2(v[ch].w, wx);
            xt[sw128_offset(xr, ch) >> 4] = o;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(bar(st::XTFULL));
        mbar_arrive(bar(st::XE00 + 2 * hh + xs));  // the X tile is not read again
        if constexpr (kHin) {
          // the state entering chunk c (the adjoint: leaving chunk c), thread =
          // state column n, all rows p
          if (live) {
            __nv_bfloat16* dst = (adj ? so.gout : so.hin) + (((int64_t)w.b * p.nc + c) * p.H + head) * kP * kN + row;
#pragma unroll
            for (int pp = 0; pp < kP; ++pp) dst[pp * kN] = __float2bfloat16_rn(hs[pp]);
          }
        }
        // h ← decay · h + S_c
        const float decay = reinterpret_cast<const float*>(sc)[128];
        if (!(ok = wait_bar(bar(st::SCFULL), cp, ctl))) break;
        tc_fence_after();
        {
          uint32_t r0[32], r1[32];
          tmem_ld32(tmem + lane_addr + 64u * hh, r0);
          tmem_ld32(tmem + lane_addr + 64u * hh + 32u, r1);
          tmem_ld_wait();
          reg_fence(r0);
          reg_fence(r1);
          tc_fence_before();
          mbar_arrive(bar(st::SCEMPTY));
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            hs[e] = fmaf(decay, hs[e], __uint_as_float(r0[e]));
            hs[32 + e] = fmaf(decay, hs[32 + e], __uint_as_float(r1[e]));
          }
        }
        dprod *= decay;
        mbar_arrive(bar(st::CSE0 + slot));
      }
      if (!ok) break;
      if (kHin && !w.last) {
        // hand the state over at the cut: stored by every thread, then the
        // flag lane raises this head's flag (the arrive releases the stores)
        float* dst = so.slot + (int64_t)(2 * w.pub + hh) * kP * kN;
#pragma unroll
        for (int pp = 0; pp < kP; ++pp) dst[pp * kN + row] = hs[pp];
        mbar_arrive(bar(st::PUB0 + hh));
      }
      if (adj && live && so.dinit && w.last) {
        // the adjoint entering chunk 0
        float* dst = so.dinit + hchain * kP * kN;
#pragma unroll
        for (int pp = 0; pp < kP; ++pp) dst[pp * kN + row] = hs[pp];
      }
      if (!kHin && live && w.s < p.nseg - 1) {
        float* dst = seg_local + (hchain * p.nseg + w.s) * kP * kN;
#pragma unroll
        for (int pp = 0; pp < kP; ++pp) dst[pp * kN + row] = hs[pp];
        if (ltid == 0) seg_decay[hchain * p.nseg + w.s] = dprod;
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, st::kTmCols);
  }
}

// h_in[s+1] = D_s · h_in[s] + h_loc[s] over the segments of each (b, h),
// h_in[0] = init_state (or 0); writes the entering state of segment s+1 where
// the fused kernel reads it, and raises the segments' flags (read by the next
// launch in stream order).  Grid (b·h, P·N / 1024); thread = 4 consecutive
// state elements, walking the segments.
__global__ void __launch_bounds__(256)
    ssd_seg_combine_kernel(const float* init, const float* seg_local, const float* seg_decay, float* seg_state,
                           uint32_t* seg_flag, int nseg) {
  // the fused kernel that consumes these states may start now: its prologue
  // and first tiles overlap this kernel, and it waits for this grid's
  // completion before it reads seg_state
  griddep_launch_dependents();
  const int64_t hc = blockIdx.x;
  const int e = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  float4 h = init ? *reinterpret_cast<const float4*>(init + hc * kP * kN + e) : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s + 1 < nseg; ++s) {
    const float d = seg_decay[hc * nseg + s];
    const float4 l = *reinterpret_cast<const float4*>(seg_local + (hc * nseg + s) * kP * kN + e);
    h.x = fmaf(d, h.x, l.x);
    h.y = fmaf(d, h.y, l.y);
    h.z = fmaf(d, h.z, l.z);
    h.w = fmaf(d, h.w, l.w);
    *reinterpret_cast<float4*>(seg_state + (hc * nseg + s) * kP * kN + e) = h;
  }
  if (blockIdx.y == 0 && threadIdx.x + 1 < (unsigned)nseg) seg_flag[hc * nseg + threadIdx.x] = 1u;
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
  return make_tma_map_bf16(m, base, B, L, W, kQ);
}

}  // namespace

// A 4-D tensor map over an fp32 [B][L][G][N] array: boxes of 32 columns (128
// bytes, 128-byte swizzle) by box_rows tokens of one group and batch row;
// coordinates (n, g, t, b).  Rows past L are clipped.
bool make_tma_map_f32_bltgn(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t G, int64_t N,
                            int box_rows) {
  auto fn = encode_fn();
  if (!fn || N % 32 != 0) return false;
  cuuint64_t dims[4] = {(cuuint64_t)N, (cuuint64_t)G, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)(N * 4), (cuuint64_t)(G * N * 4), (cuuint64_t)(L * G * N * 4)};
  cuuint32_t box[4] = {32, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 3-D tensor map over a bf16 [B][L][W] array: boxes of 64 columns (128
// bytes, 128-byte swizzle) by box_rows rows of one batch row.
bool make_tma_map_bf16(CUtensorMap* m, const void* base, int64_t B, int64_t L, int64_t W, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)W, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)(W * 2), (cuuint64_t)(L * W * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

// How a problem is cut into units, and the workspace that needs.
struct FusedPlan {
  int nseg;
  int grid;
  bool ranges;    // contiguous chunk ranges per CTA (cta_unit)
  bool two_pass;  // segment states first (ssd_states_kernel + combine), then all segments at once
  bool wants_two_pass;  // the cost model chose two passes (state size 128 only runs them)
  size_t flag_off, state_off, local_off, decay_off, memset_bytes, bytes, trace_off;
};

FusedPlan fused_plan(const Problem& p, size_t max_bytes) {
  FusedPlan pl;
  // sequences per group: head pairs, or single heads at state size 256 and
  // with the complex decay
  const bool one = p.N == 256 || p.complex_decay;
  const int64_t ppg = one ? p.H / p.G : ((p.H / p.G) + 1) / 2;
  const int64_t chains = p.B * p.G * ppg;
  const int64_t nc = (p.L + kQ - 1) / kQ;
  int sms = sm_count();
  // Test knob: SSD_FUSED_GRID caps the number of CTAs (correct for any value
  // >= 1; only the schedule changes).
  if (const char* env = getenv("SSD_FUSED_GRID")) {
    const int v = atoi(env);
    if (v >= 1) sms = std::min(sms, v);
  }
  // At least as many sequences as CTAs: one contiguous range of chunks per
  // CTA (every CTA the same number of chunks, at most one hand-off each way).
  pl.ranges = chains >= (int64_t)sms;
  // Round-robin segments (only when forced by SSD_FUSED_NSEG below, with
  // that many sequences): cost model rounds × (chunks per unit + 1/2).
  int best = 1;
  if (chains >= (int64_t)sms) {
    double best_cost = 1e30;
    for (int ns = 1; ns <= 8 && ns <= nc; ++ns) {
      const double rounds = (double)((chains * ns + sms - 1) / sms);
      const double cost = rounds * ((double)((nc + ns - 1) / ns) + 0.5);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = ns;
      }
    }
  }
  // Fewer sequences than SMs: either every sequence whole on one CTA (some SMs
  // idle), or two passes (segment states first, then every segment at once).
  // Cost in chunk times of the critical CTA: rounds × chunks per segment, the
  // two-pass schedule weighted by 1.5 for its first pass, plus one chunk per
  // round for a unit's start and end and a fixed 6 for its two extra
  // launches.  Measured on B300: 65536 tokens, 16 sequences, whole 1.74 ms ->
  // two passes (9 segments) 0.33 ms; 2048 tokens, 24 sequences of 16 chunks,
  // whole 0.070 ms -> 6 segments 0.043 ms; 4096 tokens, 128 sequences, whole.
  pl.two_pass = false;
  pl.wants_two_pass = false;
  if (chains < (int64_t)sms && nc >= 2) {
    double whole = (double)nc, best_cost = whole;
    for (int ns = 2; ns <= 64 && ns <= nc; ++ns) {
      const double rounds = (double)((chains * ns + sms - 1) / sms);
      const double cost = rounds * ((double)((nc + ns - 1) / ns) * 1.5 + 1.0) + 6.0;
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = ns;
      }
    }
    pl.two_pass = best > 1;
    // at other state sizes there are no segment-state kernels: whole
    // sequences, and for few long sequences (>= 32 chunks) the chunked path
    pl.wants_two_pass = pl.two_pass && nc >= 32;
    if (p.N != kN || p.rank_log2 > 0 || p.complex_decay) {  // (the segment-state kernel: real decay, rank 1)
      pl.two_pass = false;
      best = 1;
    }
  }
  if (const char* env = getenv("SSD_FUSED_TWOPASS")) {
    pl.two_pass = atoi(env) != 0 && chains < (int64_t)sms && nc >= 2 && p.N == kN && p.rank_log2 == 0 && !p.complex_decay;
    if (!pl.two_pass && chains < (int64_t)sms) best = 1;
    if (pl.two_pass && best == 1)
      best = (int)std::min<int64_t>({std::max<int64_t>(2, nc / 8), (int64_t)64, std::max<int64_t>(2, sms / chains)});
  }
  // Test knob: SSD_FUSED_NSEG forces the segment count (capped at the chunk
  // count so that no segment is empty).  Correct for any value; only the
  // schedule changes.
  if (const char* env = getenv("SSD_FUSED_NSEG")) {
    const int v = atoi(env);
    if (v >= 1) {
      best = (int)std::min<int64_t>(std::min<int64_t>(v, 64), std::max<int64_t>(nc, 1));
      pl.ranges = false;
    }
  }
  if (pl.ranges) {
    best = 1;  // one state slot per head: a sequence is split at most once
    pl.two_pass = false;
  }
  for (;; --best) {
    pl.nseg = best;
    if (best == 1) pl.two_pass = false;
    pl.flag_off = 256;
    const int64_t head_units = p.B * p.H * best;  // segment states are kept per head
    const size_t states = (size_t)head_units * kP * p.N * 4 * (p.complex_decay ? 2 : 1);  // (complex: Re and Im)
    const bool handoff = best > 1 || pl.ranges;
    pl.state_off = handoff ? align_up(256 + (size_t)head_units * 4, 256) : 256;
    pl.memset_bytes = pl.state_off;
    pl.local_off = pl.state_off + states;
    pl.decay_off = pl.local_off + (pl.two_pass ? states : 0);
    pl.bytes = handoff ? align_up(pl.decay_off + (pl.two_pass ? (size_t)head_units * 4 : 0), 256) : 256;
    if (pl.bytes <= max_bytes || best == 1) break;
  }
  // Without room for the hand-off states (a workspace capped below that),
  // ranges fall back to whole sequences dealt round-robin.
  if (pl.ranges && pl.bytes > max_bytes) {
    pl.ranges = false;
    pl.state_off = pl.memset_bytes = pl.local_off = pl.decay_off = 256;
    pl.bytes = 256;
  }
  // SSD_FUSED_TRACE=1: role timestamps of CTA 0 in the last bytes of the workspace
  pl.trace_off = 0;
  if (const char* env = getenv("SSD_FUSED_TRACE")) {
    if (atoi(env) == 1 && max_bytes == SIZE_MAX) {
      pl.trace_off = align_up(pl.bytes, 256);
      pl.bytes = pl.trace_off + ((size_t)kTraceChunks * kTraceEvents + 6 * kTraceCtas) * 8;
    }
  }
  pl.grid = (int)std::min<int64_t>(chains * pl.nseg, sms);
  return pl;
}

// ---------------------------------------------------------------- static scratch
// Scratch for ssd_fwd_noalloc: a fixed device array in the library image, so
// callers that must not allocate device memory still have somewhere for the
// fused kernel's workspace.  Every GPU that loads the library holds it until
// the process exits.
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
  return p.io == SSD_DTYPE_BF16 && p.P == kP && (p.N == 256 || p.N == 128 || p.N == 64 || p.N == 16) &&
         (p.Q_req == 0 || p.Q_req == kQ) && p.B * p.H < (int64_t(1) << 24) && p.L < (int64_t(1) << 30) &&
         encode_fn() != nullptr;
}

bool fused_preferred(const Problem& p) {
  if (!fused_supported(p)) return false;
  // state sizes 64 and 16 have no two-pass schedule: where it would pay off
  // (few long sequences), the chunked path keeps more SMs busy
  return p.N == kN || !fused_plan(p, SIZE_MAX).wants_two_pass;
}

size_t fused_workspace_bytes(const Problem& p, size_t max_bytes) { return fused_plan(p, max_bytes).bytes; }

cudaError_t launch_fused(const Problem& p, void* workspace, cudaStream_t s, size_t max_bytes) {
  CUtensorMap tx, tb, tc, ty, tz;
  // dstate below 64 (16): 4-D [B][L][G][N] maps whose 64-column boxes read
  // zeros past N, so the kernel of state size 64 serves it unchanged
  const bool narrow = p.N < 64;
  auto map_bc = [&](CUtensorMap* m, const void* base) {
    return narrow ? make_tma_map_bf16_narrow(m, base, p.B, p.L, p.G, p.N, kQ)
                  : make_map(m, base, p.B, p.L, p.G * p.N);
  };
  if (!make_map(&tx, p.x, p.B, p.L, p.H * kP) || !map_bc(&tb, p.Bm) || !map_bc(&tc, p.Cm) ||
      !make_map(&ty, p.y, p.B, p.L, p.H * kP) || (p.z && !make_map(&tz, p.z, p.B, p.L, p.H * kP)))
    return cudaErrorInvalidValue;
  const FusedPlan pl = fused_plan(p, max_bytes);
  const bool delta = p.dt_bias != nullptr || p.dt_softplus != 0;
  using KernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, FusedParams);
  KernelFn kernel;
  uint32_t smem;
  // (retrieval rank comes through its own entry point: no Δ pre-processing, no gate)
  const bool rank = p.rank_log2 > 0;
  if (rank && (delta || p.z)) return cudaErrorInvalidValue;
  // (the complex decay comes through its own entry point: state size 128, no
  // Δ pre-processing, gate or rank)
  const bool rot = p.complex_decay;
  if (rot && (delta || p.z || rank || p.N != 128 || !p.theta)) return cudaErrorInvalidValue;
  if (rot) {
    kernel = ssd_fused_kernel<false, false, 128, false, true>;
    smem = Lay<128, true>::kSmemAlloc;
  } else if (p.N == 128) {
    kernel = rank ? ssd_fused_kernel<false, false, 128, true>
           : p.z  ? (delta ? ssd_fused_kernel<true, true, 128> : ssd_fused_kernel<false, true, 128>)
                  : (delta ? ssd_fused_kernel<true, false, 128> : ssd_fused_kernel<false, false, 128>);
    smem = Lay<128>::kSmemAlloc;
  } else if (p.N == 256) {
    kernel = rank ? ssd_fused_kernel<false, false, 256, true>
           : p.z  ? (delta ? ssd_fused_kernel<true, true, 256> : ssd_fused_kernel<false, true, 256>)
                  : (delta ? ssd_fused_kernel<true, false, 256> : ssd_fused_kernel<false, false, 256>);
    smem = Lay<256>::kSmemAlloc;
  } else {
    kernel = rank ? ssd_fused_kernel<false, false, 64, true>
           : p.z  ? (delta ? ssd_fused_kernel<true, true, 64> : ssd_fused_kernel<false, true, 64>)
                  : (delta ? ssd_fused_kernel<true, false, 64> : ssd_fused_kernel<false, false, 64>);
    smem = Lay<64>::kSmemAlloc;
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // the error word and the segment flags start at zero on every call (in
  // two-pass mode the states kernel clears them)
  if (!pl.two_pass && (e = cudaMemsetAsync(workspace, 0, pl.memset_bytes, s)) != cudaSuccess) return e;
  char* ws = static_cast<char*>(workspace);
  FusedParams fp;
  fp.dt = p.dt;
  fp.A = p.A;
  fp.D = p.D;
  fp.init = p.init;
  fp.final_state = p.final_state;
  fp.publish = pl.two_pass ? 0 : 1;
  fp.dt_bias = p.dt_bias;
  fp.dt_softplus = p.dt_softplus;
  fp.B = (int32_t)p.B;
  fp.L = (int32_t)p.L;
  fp.H = (int32_t)p.H;
  fp.G = (int32_t)p.G;
  fp.nc = (int32_t)((p.L + kQ - 1) / kQ);
  fp.heads_per_chain = (p.N == 256 || rot) ? 1 : 2;
  fp.pairs_per_group = (int32_t)((p.N == 256 || rot) ? p.H / p.G : ((p.H / p.G) + 1) / 2);
  fp.chains = (int32_t)(p.B * p.G * fp.pairs_per_group);
  fp.nseg = pl.nseg;
  fp.units = fp.chains * pl.nseg;
  fp.ranges = pl.ranges ? 1 : 0;
  fp.nstate = (int32_t)p.N;
  fp.Ltok = (int32_t)(p.L >> p.rank_log2);
  fp.rank_log2 = p.rank_log2;
  fp.narrow = narrow ? 1 : 0;
  fp.theta = p.theta;
  fp.init_im = p.init_im;
  fp.final_im = p.final_im;
  fp.pdl = pl.two_pass ? 1 : 0;
  fp.zero_words = pl.two_pass ? (uint32_t)(pl.memset_bytes / 16) : 0u;
  fp.err = reinterpret_cast<int32_t*>(ws);
  fp.seg_flag = reinterpret_cast<uint32_t*>(ws + pl.flag_off);
  fp.seg_state = (pl.nseg > 1 || pl.ranges) ? reinterpret_cast<float*>(ws + pl.state_off) : nullptr;
  // Every device wait gives up after this long (2 s).  Test knobs for the
  // failure path: SSD_FUSED_TIMEOUT_MS shortens the limit, and
  // SSD_FUSED_TEST_NO_FLAGS=1 never raises the hand-off flags, so that the
  // units waiting on them run out of time and the call reports
  // SSD_ERR_TIMEOUT through ssd_workspace_status().
  fp.timeout_ns = 2000000000ull;
  if (const char* env = getenv("SSD_FUSED_TIMEOUT_MS")) {
    const long v = atol(env);
    if (v >= 1 && v <= 2000) fp.timeout_ns = (uint64_t)v * 1000000ull;
  }
  fp.test_no_flags = 0;
  if (const char* env = getenv("SSD_FUSED_TEST_NO_FLAGS")) fp.test_no_flags = atoi(env) == 1 ? 1 : 0;
  fp.trace = pl.trace_off ? reinterpret_cast<long long*>(ws + pl.trace_off) : nullptr;
  if (fp.trace && (e = cudaMemsetAsync(fp.trace, 0, ((size_t)kTraceChunks * kTraceEvents + 6 * kTraceCtas) * 8, s)) !=
                      cudaSuccess)
    return e;
  if (pl.two_pass) {
    float* local = reinterpret_cast<float*>(ws + pl.local_off);
    float* decay = reinterpret_cast<float*>(ws + pl.decay_off);
    auto states = delta ? ssd_states_kernel<true> : ssd_states_kernel<false>;
    if ((e = cudaFuncSetAttribute(states, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st::kSmemAlloc)) !=
        cudaSuccess)
      return e;
    states<<<pl.grid, 384, st::kSmemAlloc, s>>>(tx, tb, tx, tb, fp, local, decay, SeqOut{});
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    static_assert(kP * kN % 1024 == 0, "combine grid");
    ssd_seg_combine_kernel<<<dim3((unsigned)(p.B * p.H), kP * kN / 1024), 256, 0, s>>>(
        p.init, local, decay, fp.seg_state, fp.seg_flag, pl.nseg);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // CTAs wait on states handed over by other CTAs of the same launch (ranges,
  // or segments published within the launch): launched as a cooperative
  // grid, so that either all of its CTAs are resident at once or the launch
  // fails with an error, instead of a wait that cannot end.
  const bool handoffs = fp.publish && (pl.ranges || pl.nseg > 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (handoffs) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    // two-pass mode: a programmatic dependent of the combine kernel (see pdl)
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = (handoffs || fp.pdl) ? 1 : 0;
  const CUtensorMap& tzz = p.z ? tz : tx;
  return cudaLaunchKernelEx(&cfg, kernel, tx, tb, tc, ty, tzz, fp);
}

bool states_hin_supported(const Problem& p) {
  return p.io == SSD_DTYPE_BF16 && p.P == kP && p.N == kN && p.Q == kQ && p.B * p.H < (int64_t(1) << 24) &&
         p.L < (int64_t(1) << 30) && encode_fn() != nullptr;
}

int states_walks(const Problem& p) { return (int)(2 * p.B * p.G * (((p.H / p.G) + 1) / 2)); }

// The states entering every chunk (forward) and the adjoint leaving every
// chunk, both bf16 [B][nc][H][P][N], and dinit, for the backward pass: one
// launch of the states kernel over 2 · (head-pair sequences) walks, the
// forward ones first, cut into one contiguous range of steps per CTA (the
// fp32 state on chip, handed over once at each cut through `flags`, zeroed
// by the caller, and `slots`).  Launched cooperatively: CTAs wait on each
// other's hand-offs.  Its bounded waits record SSD_ERR_TIMEOUT in *err.
cudaError_t launch_states_walks(const Problem& p, void* hin, const void* dy, const float* dfinal, float* dinit,
                                void* gout, uint32_t* flags, float* slots, int32_t* err, cudaStream_t s) {
  if (!states_hin_supported(p)) return cudaErrorInvalidValue;
  if (p.B == 0 || p.L == 0) return cudaSuccess;
  CUtensorMap tx, tb, tdy, tc;
  if (!make_map(&tx, p.x, p.B, p.L, p.H * kP) || !make_map(&tb, p.Bm, p.B, p.L, p.G * p.N) ||
      !make_map(&tdy, dy, p.B, p.L, p.H * kP) || !make_map(&tc, p.Cm, p.B, p.L, p.G * p.N))
    return cudaErrorInvalidValue;
  FusedParams fp = {};
  fp.dt = p.dt;
  fp.A = p.A;
  fp.init = p.init;
  fp.B = (int32_t)p.B;
  fp.L = (int32_t)p.L;
  fp.H = (int32_t)p.H;
  fp.G = (int32_t)p.G;
  fp.nc = (int32_t)((p.L + kQ - 1) / kQ);
  fp.heads_per_chain = 2;
  fp.pairs_per_group = (int32_t)(((p.H / p.G) + 1) / 2);
  fp.chains = (int32_t)(p.B * p.G * fp.pairs_per_group);
  fp.nseg = 1;
  fp.units = 2 * fp.chains;
  fp.nstate = (int32_t)p.N;
  fp.Ltok = (int32_t)p.L;
  fp.err = err;
  fp.timeout_ns = 2000000000ull;
  SeqOut so;
  so.hin = static_cast<__nv_bfloat16*>(hin);
  so.gout = static_cast<__nv_bfloat16*>(gout);
  so.dfinal = dfinal;
  so.dinit = dinit;
  so.units_fwd = fp.chains;
  so.flag = flags;
  so.slot = slots;
  auto kernel = ssd_states_kernel<false, 1>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st::kSmemAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min<int64_t>(fp.units, sm_count()));  // ranges at least one walk long
  cfg.blockDim = dim3(384);
  cfg.dynamicSmemBytes = st::kSmemAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tx, tb, tdy, tc, fp, (float*)nullptr, (float*)nullptr, so);
}

}  // namespace ssd
