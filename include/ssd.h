/*
 * ssd.h -- C ABI of the B300 (sm_103a) SSD selective-scan forward library.
 *
 * The operation.  For every batch row b and head h, with Δ_t = dt[b,t,h],
 * α_t = exp(Δ_t·A[h]) and g = h / (nheads/ngroups), the library computes
 *
 *     h_t[p][n] = α_t · h_{t-1}[p][n] + Δ_t · x[b,t,h,p] · Bm[b,t,g,n]
 *     y[b,t,h,p] = Σ_n Cm[b,t,g,n] · h_t[p][n] + D[h] · x[b,t,h,p]
 *
 * with h_{-1} = init_state[b,h] (zeros when absent) and
 * final_state[b,h] = h_{L-1}.  This is the discretised selective SSM of the
 * page "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of SSM)":
 * §2.1.2 (Euler/ZOH step h_t = e^{Δ_t A_t} h_{t-1} + Δ_t B_t x_t, forget gate
 * α_t, input gate γ_t = Δ_t, boxed recurrence, output y_t = C_tᵀ h_t) plus the
 * skip term D x of §2.1.1, with A a real scalar per head (§2.3.1).  It is
 * evaluated in its chunked dual form: inside a chunk of Q tokens the masked
 * matrix product Y = (L ⊙ C Bᵀ) X of §2.2.1 (mask L_ij = ∏_{k=j+1}^{i} α_k),
 * across chunks the same recurrence lifted to chunk granularity (the block
 * decomposition of the mask figure in §2.2.2).  Heads share B/C in G
 * contiguous groups ("Transformers are SSMs", §2.1, grouped heads).
 *
 * Layouts.  Every tensor is dense, row-major, in the order written:
 *     x, y         [batch][seqlen][nheads][headdim]      io dtype
 *     dt           [batch][seqlen][nheads]               fp32, Δ ≥ 0 (after softplus)
 *     A            [nheads]                              fp32, A ≤ 0
 *     Bm, Cm       [batch][seqlen][ngroups][dstate]      io dtype
 *     D            [nheads]                              fp32 (NULL: no skip term)
 *     init_state,
 *     final_state  [batch][nheads][headdim][dstate]      fp32
 * The io dtype is fp32 or bf16; all accumulation and the state are fp32.
 *
 * Ownership.  Every pointer is device memory owned by the caller and must
 * be 16-byte aligned.  The library allocates no device memory: scratch
 * space is the caller's `workspace` (size from ssd_fwd_workspace_size).
 * Outputs must not overlap inputs, except that final_state may equal
 * init_state exactly (in-place state update).
 *
 * Streams and errors.  Every call is asynchronous on `stream` (a
 * cudaStream_t passed as void*; NULL = the legacy default stream).  Arguments
 * are validated on the host before anything is launched; on failure nothing
 * is launched and a status code is returned.  Launch failures map to
 * SSD_ERR_CUDA.  Faults during device execution surface at the caller's next
 * synchronisation, as usual for CUDA.  No C++ exception crosses this ABI.
 * ssd_last_error_message() describes the last failure on the calling thread.
 */
#ifndef SSD_SCAN_FWD_SSD_H_
#define SSD_SCAN_FWD_SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_ABI_VERSION 1

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1, /* null required pointer, bad size, overlap, misalignment */
  SSD_ERR_UNSUPPORTED = 2, /* valid problem the library has no kernel for */
  SSD_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  SSD_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  SSD_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see ssd_workspace_status) */
} ssd_status;

typedef enum { SSD_DTYPE_F32 = 0, SSD_DTYPE_BF16 = 1 } ssd_dtype;

typedef enum {
  SSD_ALGO_AUTO = 0,    /* fused tensor-core kernel when the shape allows it, else chunked */
  SSD_ALGO_CHUNKED = 1, /* the four step kernels below, in order (chunk states and
                           outputs on tcgen05 for bf16, headdim 64, dstate 16-256
                           at chunk 128; fp32 CUDA cores otherwise) */
  SSD_ALGO_FUSED = 2    /* one persistent tcgen05/TMA kernel, state kept on chip (bf16 io,
                           headdim 64, dstate 16, 64 or 128) */
} ssd_algo;

typedef struct {
  int64_t batch;      /* B  >= 0 */
  int64_t seqlen;     /* L  >= 0 */
  int64_t nheads;     /* H  >= 1 */
  int64_t headdim;    /* P  in [1, 256] */
  int64_t ngroups;    /* G  >= 1, divides H */
  int64_t dstate;     /* N  in [1, 256] */
  int32_t io_dtype;   /* ssd_dtype of x, Bm, Cm, y */
  int32_t algo;       /* ssd_algo */
  int64_t chunk_size; /* Q for the chunked path: 32, 64 or 128.  0 = default:
                         128 where the chunk states and outputs run on the tensor
                         cores (bf16 io, headdim 64, dstate 16, 64, 128 or 256), else
                         64 */
  const void* x;
  const float* dt;
  const float* A;
  const void* Bm;
  const void* Cm;
  const float* D;          /* may be NULL: no skip term */
  const float* init_state; /* may be NULL: zero initial state */
  void* y;
  float* final_state;      /* may be NULL: not written */
  void* workspace;         /* device scratch, >= ssd_fwd_workspace_size() bytes, 256-B aligned */
  size_t workspace_bytes;
} ssd_fwd_args;

/* ABI version of the loaded library (SSD_ABI_VERSION it was built with). */
int ssd_abi_version(void);

/* Bytes of workspace ssd_fwd needs for these arguments (pointers are not
 * inspected).  Returns (size_t)-1 when the shape or options are invalid or
 * unsupported. */
size_t ssd_fwd_workspace_size(const ssd_fwd_args* args);

/* The whole forward pass: y and (optionally) final_state. */
ssd_status ssd_fwd(const ssd_fwd_args* args, void* stream);

/* The status the last call that used `workspace` left on the device:
 * SSD_OK, or SSD_ERR_TIMEOUT when one of its kernels' bounded device-side
 * waits gave up (that kernel then stops, releases what it holds and leaves
 * its outputs unspecified; the CUDA context stays usable).  Every entry point
 * that takes a workspace (ssd_fwd, ssd_fwd_ex, ssd_fwd_host, ssd_fwd_rot,
 * ssd_bwd) clears the word at the start of its workspace when it is called
 * and its kernels write SSD_ERR_TIMEOUT there: the fused kernel's waits on
 * other CTAs' state hand-offs and on its own loads and MMAs, and the
 * tensor-core kernels' waits on their own loads and MMAs.  Synchronises
 * `stream`, then reads that word; call it before the workspace is reused. */
ssd_status ssd_workspace_status(const void* workspace, void* stream);

/* Static description of a status code. */
const char* ssd_status_string(ssd_status status);

/* Description of the last failure on the calling thread ("" if none). */
const char* ssd_last_error_message(void);

/* The forward pass with the steps that surround the scan in a Mamba block
 * (page "从 SSM 的长期记忆问题，到 Mamba 的选择性机制与硬件感知扫描", the
 * paragraphs on the selective SSM and on the Mamba block): Δ is formed from a
 * per-head parameter plus the input-dependent part through τ_Δ, and the scan's
 * output is gated.  Here, with base.dt holding the raw input-dependent part,
 *
 *     Δ[b,t,h] = softplus(dt[b,t,h] + dt_bias[h])   (dt_softplus = 1)
 *     Δ[b,t,h] = dt[b,t,h] + dt_bias[h]             (dt_softplus = 0; must be >= 0)
 *     y        = scan(Δ, ...) · silu(z),  silu(z) = z / (1 + e^{-z})   (z != NULL)
 *
 * softplus(v) = log(1 + e^v).  The page names τ_Δ and the gate without
 * formulas; softplus and the SiLU gate are this library's reading.  The state
 * (final_state) is the scan's, never gated.  Same conventions and workspace as
 * ssd_fwd (ssd_fwd_ex_workspace_size equals ssd_fwd_workspace_size(&base)). */
typedef struct {
  ssd_fwd_args base;      /* the scan's arguments; base.dt is the raw dt */
  const float* dt_bias;   /* [nheads] fp32, may be NULL: no bias */
  int32_t dt_softplus;    /* 0 or 1 */
  int32_t reserved;       /* must be 0 */
  const void* z;          /* [batch][seqlen][nheads][headdim] io dtype, may be NULL: no gate */
} ssd_fwd_ex_args;

size_t ssd_fwd_ex_workspace_size(const ssd_fwd_ex_args* args);
ssd_status ssd_fwd_ex(const ssd_fwd_ex_args* args, void* stream);

/* The forward pass on HOST buffers.  args->x, dt, A, Bm, Cm, D, init_state,
 * y and final_state are host pointers (page-locked memory lets the copies
 * overlap the compute; pageable memory works but serialises them);
 * args->workspace is DEVICE memory of at least
 * ssd_fwd_host_workspace_size(args) bytes, 256-byte aligned.  The library
 * cuts the problem into groups and pipelines them through two device staging
 * slots: copies in on one stream of its own, the forward pass (as ssd_fwd,
 * same algo choice) on `stream`, copies out on another stream of its own, so
 * that the copies of one group overlap the compute of the next.  Sequences
 * of at least 512 tokens are cut along the tokens into up to 16 segments of
 * whole 128-token chunks (every batch row in each group; the state passes
 * from one segment's forward pass to the next in fp32 device buffers),
 * shorter ones into four groups of batch rows.
 * The call is asynchronous: everything it enqueues is ordered after the work
 * already on `stream`, and `stream` waits for the last copy out, so y and
 * final_state are ready once `stream` is synchronised.  Its two copy streams
 * and its events are created on the first call on a device and kept until
 * the process exits; calls on one device are serialised while they enqueue.
 * It allocates no memory.  The first word of the workspace collects the
 * status of every group's forward pass (ssd_workspace_status).  The host
 * buffers must stay valid (and, for the outputs, unread) until then.  Not
 * part of the pages: a convenience for callers whose data live in host
 * memory. */
size_t ssd_fwd_host_workspace_size(const ssd_fwd_args* args);
ssd_status ssd_fwd_host(const ssd_fwd_args* args, void* stream);

/* Allocation-free variant of ssd_fwd, for callers that cannot allocate device
 * memory themselves: for example code whose device memory is all owned by a
 * host framework's pool (no raw cudaMalloc allowed), or latency-critical loops
 * where a cudaMalloc/cudaFree could synchronise the device.  It runs the fused
 * kernel (bf16 io, headdim 64, dstate 16, 64 or 128; algo AUTO or FUSED) and takes its
 * scratch from a fixed 1 MiB device array inside the library instead of
 * args->workspace (ignored).  Inputs and outputs are still the caller's.
 * Nothing is rejected for its size: where the hand-off states of the usual
 * schedule (one contiguous chunk range per CTA, or sequences cut into
 * segments) would not fit in 1 MiB, every sequence runs whole on one CTA,
 * which is slower when there are about as many sequences as SMs or fewer
 * (for example the 2.7B-shaped layer, 320 heads × 32 KB of states: 160
 * head-pair sequences on 148 SMs).  The first call on a device resolves the
 * array's device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture.  Every call on a device shares the
 * one array, which keeps the last call's contents (the call clears what must
 * start at zero): calls that overlap on the GPU (different streams, no
 * ordering) race on it.  It allocates nothing: no cudaMalloc, cudaFree or
 * allocating library routine.  The pages have no counterpart of this entry
 * point; it is part of the library's interface only. */
ssd_status ssd_fwd_noalloc(const ssd_fwd_args* args, void* stream);

/* The status the last ssd_fwd_noalloc call on the current device left in the
 * fixed array (SSD_OK or SSD_ERR_TIMEOUT, as ssd_workspace_status).
 * Synchronises `stream`; call it before the next ssd_fwd_noalloc call, which
 * clears the word.  No counterpart on the pages either. */
ssd_status ssd_fwd_noalloc_status(void* stream);

/* ------------------------------------------------------------------------
 * Retrieval rank R > 1 (MIMO): the page "状态空间模型的对角等价：检索秩与选择性
 * 扩展新解", section "从 MIMO 到 HybridMamba", defines the retrieval rank as
 * the number of independent value channels written and read in parallel at a
 * local interface, with an independent value routed per rank and SISO
 * (R = 1) recovered exactly; it prints no formula.  This library's reading:
 * per token t and head, R ranks r with their own x_t^(r), B_t^(r), C_t^(r)
 * share the token's decay, the update writes all R values, each rank reads
 * its own output from the updated state:
 *
 *     h_t     = α_t · h_{t-1} + Δ_t · Σ_r x_t^(r) · B_t^(r)ᵀ
 *     y_t^(r) = h_t · C_t^(r) + D[h] · x_t^(r)
 *
 * Layouts: base.seqlen = L tokens; x, y [batch][seqlen][rank][nheads][headdim];
 * Bm, Cm [batch][seqlen][rank][ngroups][dstate]; dt [batch][seqlen][nheads]
 * (one Δ per token); A, D, states as for ssd_fwd.  In the chunked form the
 * R rows of a token are consecutive rows of a chunk; inside a chunk the mask
 * keeps (row i, row j) when token(j) ≤ token(i), with the decay between
 * tokens.  Runs the fused kernel only: bf16 io, headdim 64, dstate 16, 64,
 * 128 or 256, rank 1, 2, 4 or 8 (SSD_ERR_UNSUPPORTED otherwise); base.algo
 * AUTO or FUSED.  Same conventions and status word as ssd_fwd.
 * ------------------------------------------------------------------------ */
typedef struct {
  ssd_fwd_args base;  /* sizes and pointers as above; base.seqlen counts tokens */
  int64_t rank;       /* R: 1, 2, 4 or 8 */
} ssd_fwd_mimo_args;

size_t ssd_fwd_mimo_workspace_size(const ssd_fwd_mimo_args* args);
ssd_status ssd_fwd_mimo(const ssd_fwd_mimo_args* args, void* stream);

/* ------------------------------------------------------------------------
 * Recurrent step (inference).  One token per (batch row, head): the same
 * recurrence, evaluated directly rather than in its chunked dual form
 * ("Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of SSM)", the boxed
 * recurrence of §2.1.2 with the skip term of §2.1.1; §2.2.2: at inference the
 * dual form switches back to this recurrence, with an O(1) state):
 *
 *     state[b,h][p][n] = exp(dt[b,h]·A[h]) · state[b,h][p][n] + dt[b,h] · x[b,h,p] · Bm[b,g,n]
 *     y[b,h,p]         = Σ_n Cm[b,g,n] · state[b,h][p][n] + D[h] · x[b,h,p]
 *
 * with g = h / (nheads/ngroups) and the state updated in place.  Calling it
 * for t = 0..L-1 on the rows of a sequence gives the y and final_state of
 * ssd_fwd over those L tokens (up to rounding).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t batch;     /* B >= 0 (0: nothing to do) */
  int64_t nheads;    /* H >= 1 */
  int64_t headdim;   /* P in [1, 256] */
  int64_t ngroups;   /* G >= 1, divides H */
  int64_t dstate;    /* N in [1, 256] */
  int32_t io_dtype;  /* ssd_dtype of x, Bm, Cm, y */
  int32_t reserved;  /* must be 0 */
  const void* x;     /* [batch][nheads][headdim]  io dtype */
  const float* dt;   /* [batch][nheads]           fp32, Δ >= 0 */
  const float* A;    /* [nheads]                  fp32 */
  const void* Bm;    /* [batch][ngroups][dstate]  io dtype */
  const void* Cm;    /* [batch][ngroups][dstate]  io dtype */
  const float* D;    /* [nheads] fp32, may be NULL: no skip term */
  float* state;      /* [batch][nheads][headdim][dstate] fp32, read and overwritten */
  void* y;           /* [batch][nheads][headdim]  io dtype, written */
} ssd_step_args;

/* One recurrent step.  Same conventions as ssd_fwd: device pointers owned by
 * the caller, 16-byte aligned; y must not overlap any input or the state;
 * the state may not overlap the other inputs.  Needs no workspace. */
ssd_status ssd_step(const ssd_step_args* args, void* stream);

/* ------------------------------------------------------------------------
 * The complex (rotational) decay of Mamba-3 ("Mamba-3 深度剖析 - 02",
 * §2.3: a real decay cannot rotate or oscillate, e^{iθ} = cos θ + i sin θ can;
 * the parity task as the example).  This library's reading: every token and
 * head has a rotation angle θ[b,t,h] next to Δ, and
 *     α_t = exp(Δ_t·A[h]) · (cos θ_t + i sin θ_t)
 *     h_t = α_t · h_{t-1} + Δ_t · x_t · B_tᵀ        (complex P×N state)
 *     y_t = Re(h_t) · C_t + D[h] · x_t
 * θ = 0 gives ssd_fwd.  Chunked form: inside a chunk the mask becomes
 * exp(cs_i − cs_j)·cos(φ_i − φ_j) with φ the in-chunk sums of θ; across
 * chunks the complex state is carried (fp32).  Paths: bf16 io, headdim 64,
 * dstate 128, chunk_size 0 or 128 and base.algo AUTO or FUSED: the fused
 * kernel, one head per CTA with the complex state kept on chip (its Re and Im
 * parts rounded to bf16 only as MMA operands); base.algo FUSED on any other
 * problem: SSD_ERR_UNSUPPORTED.  Otherwise (or base.algo CHUNKED) the chunked
 * path: bf16 io with headdim 64 and dstate 16, 64, 128 or 256 at chunk 128
 * (the default there): chunk states and chunk outputs on the tensor cores
 * (bf16 operands, fp32 accumulation, the entering states rounded to bf16 as
 * operands); otherwise fp32 CUDA cores, chunk 64 by default.  The workspace
 * size depends on the path (ssd_fwd_rot_workspace_size follows the same
 * rule).  The real parts of the initial and final states are
 * base.init_state / base.final_state, the imaginary parts the fields below.
 * ------------------------------------------------------------------------ */
typedef struct {
  ssd_fwd_args base;
  const float* theta;          /* [batch][seqlen][nheads] fp32, required */
  const float* init_state_im;  /* [batch][nheads][headdim][dstate] fp32, NULL: zero */
  float* final_state_im;       /* [batch][nheads][headdim][dstate] fp32, NULL: not written */
} ssd_fwd_rot_args;

size_t ssd_fwd_rot_workspace_size(const ssd_fwd_rot_args* args);
ssd_status ssd_fwd_rot(const ssd_fwd_rot_args* args, void* stream);

/* ------------------------------------------------------------------------
 * The backward pass: the gradient of  Σ dy ⊙ y + Σ dfinal ⊙ final_state
 * with respect to every input of ssd_fwd, for the recurrence above
 * ("Mamba-3 深度剖析 - 02", §2.1.2, plus the skip term of §2.1.1).  The states
 * are recomputed, not stored by the forward call (the page "从 SSM 的长期记忆
 * 问题，到 Mamba 的选择性机制与硬件感知扫描", paragraph on the hardware-aware
 * scan: recomputation in the backward pass).  With G_t the gradient of the
 * scalar with respect to h_t:
 *     dx_t  = D dy_t + Δ_t G_t B_t
 *     dΔ_t  = x_tᵀ G_t B_t + A[h] <G_t, α_t h_{t-1}>          (ddt: w.r.t. Δ = dt)
 *     dA[h] = Σ_{b,t} Δ_t <G_t, α_t h_{t-1}>
 *     dBm   = Σ_{heads of the group} Δ_t G_tᵀ x_t,   dCm = Σ_{heads} h_tᵀ dy_t
 *     dD[h] = Σ_{b,t} dy_t·x_t,   dinit = α_0 G_0
 * Chunked form.  bf16 with headdim 64 and dstate 128: chunk length 128, the
 * per-chunk contractions on the tensor cores (bf16 operands, fp32
 * accumulation, the decay masks rounded to bf16 as operands); otherwise
 * chunk length 64, fp32 arithmetic on CUDA cores.
 * ------------------------------------------------------------------------ */
typedef struct {
  ssd_fwd_args fwd;     /* the forward call's sizes, io_dtype, x, dt (Δ), A, Bm, Cm, D,
                           init_state; y, final_state and algo are ignored; chunk_size
                           0 (default: 128 where the tensor-core path applies,
                           else 64), 64, or 128 (bf16, headdim 64, dstate 128
                           only; SSD_ERR_UNSUPPORTED otherwise); workspace,
                           workspace_bytes: scratch */
  const void* dy;       /* [batch][seqlen][nheads][headdim] io dtype, required */
  const float* dfinal;  /* [batch][nheads][headdim][dstate] fp32, NULL: zero */
  void* dx;             /* [batch][seqlen][nheads][headdim] io dtype, written */
  float* ddt;           /* [batch][seqlen][nheads] fp32, written */
  float* dA;            /* [nheads] fp32, written */
  void* dBm;            /* [batch][seqlen][ngroups][dstate] io dtype, written */
  void* dCm;            /* [batch][seqlen][ngroups][dstate] io dtype, written */
  float* dD;            /* [nheads] fp32, written; may be NULL */
  float* dinit;         /* [batch][nheads][headdim][dstate] fp32, written; may be NULL */
} ssd_bwd_args;

/* Scratch bytes ssd_bwd needs ((size_t)-1 on invalid arguments). */
size_t ssd_bwd_workspace_size(const ssd_bwd_args* args);

/* The gradients.  Same conventions as ssd_fwd: device pointers owned by the
 * caller, 16-byte aligned, outputs overlapping neither the inputs nor each
 * other; validated before any launch.  headdim up to 128 (SSD_ERR_UNSUPPORTED
 * above).  dBm and dCm are accumulated in fp32 and rounded once to the io
 * dtype. */
ssd_status ssd_bwd(const ssd_bwd_args* args, void* stream);

/* ------------------------------------------------------------------------
 * The four steps of the chunked path, exported one by one so that each can
 * be checked against the oracle's chunked intermediates and composed by the
 * caller.  They read the shape, dtype and io pointers from `args` (its algo
 * and workspace fields are ignored) and use chunk length `chunk`
 * (32, 64 or 128), nc = ceil(seqlen / chunk).  Intermediate layouts:
 *     dA_cs, dt_chunked   [batch][nheads][nc][chunk]          fp32
 *     states              [batch][nc][nheads][headdim][dstate] fp32
 * Positions past seqlen in the last chunk carry Δ = 0 (α = 1, no input).
 * ------------------------------------------------------------------------ */

/* Step 1, chunk_cumsum: log α_t = Δ_t·A[h] and its inclusive running sum
 * inside each chunk, cs_i = Σ_{k≤i} Δ_k A[h] ("Mamba-3 深度剖析 - 02", §2.1.2:
 * α_t = e^{Δ_t A_t}; §2.2.1: products of α in the mask become differences of
 * these sums).  Writes dA_cs and dt_chunked (Δ re-laid out per chunk, 0 past
 * seqlen). */
ssd_status ssd_chunk_cumsum(const ssd_fwd_args* args, int64_t chunk, float* dA_cs,
                            float* dt_chunked, void* stream);

/* Step 2, chunk_state: the state each chunk produces from zero,
 * S_c[p][n] = Σ_i exp(cs_{Q-1} − cs_i) · Δ_i · x_i[p] · Bm_i[n]
 * (§2.2.1's mask restricted to "from token i to the chunk end").  Writes
 * states. */
ssd_status ssd_chunk_state(const ssd_fwd_args* args, int64_t chunk, const float* dA_cs,
                           const float* dt_chunked, float* states, void* stream);

/* Step 3, state_passing: the recurrence of §2.1.2 lifted to chunks,
 * h_in[0] = init_state, h_in[c+1] = exp(cs_{c,Q-1}) · h_in[c] + S_c.
 * Overwrites states[c] with h_in[c] (the state entering chunk c) and writes
 * args->final_state = h_in[nc] when it is not NULL. */
ssd_status ssd_state_passing(const ssd_fwd_args* args, int64_t chunk, const float* dA_cs,
                             float* states, void* stream);

/* Step 4, chunk_scan: per chunk,
 * y_i = Σ_{j≤i} (C_i·B_j) exp(cs_i − cs_j) Δ_j x_j + exp(cs_i) C_iᵀ h_in[c] + D x_i
 * (§2.2.1's Y = (L ⊙ C Bᵀ) X inside the chunk, the state read-out
 * y_t = C_tᵀ h_t of §2.1.2 for the carried state, the skip term of §2.1.1).
 * Reads states as written by step 3; writes args->y. */
ssd_status ssd_chunk_scan(const ssd_fwd_args* args, int64_t chunk, const float* dA_cs,
                          const float* dt_chunked, const float* states, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_SCAN_FWD_SSD_H_ */
