// api.cu -- the C ABI: argument validation, workspace sizing, dispatch.
//
// Nothing here computes the scan; it checks a call before any launch and
// hands a validated Problem to the kernels of chunked.cu / fused.cu on the
// caller's stream.

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"

#define SSD_API extern "C" __attribute__((visibility("default")))

namespace ssd {
namespace {

thread_local char g_err[512] = "";

ssd_status fail(ssd_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

ssd_status cuda_fail(cudaError_t e, const char* what) {
  return fail(SSD_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int64_t kMaxDim = int64_t(1) << 31;

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
  if (a < 0 || b < 0) return false;
  if (a != 0 && b > (int64_t(1) << 62) / a) return false;
  *out = a * b;
  return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Span {
  const void* p;
  size_t n;
  const char* name;
};

bool overlaps(const Span& a, const Span& b) {
  if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
  return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Shape and option checks (no pointers).  Fills sizes of the problem.
ssd_status check_shape(const ssd_fwd_args* a, int64_t chunk, Problem* pr) {
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  if (a->batch < 0 || a->seqlen < 0) return fail(SSD_ERR_INVALID_ARG, "batch and seqlen must be >= 0");
  if (a->nheads < 1 || a->ngroups < 1 || a->headdim < 1 || a->dstate < 1)
    return fail(SSD_ERR_INVALID_ARG, "nheads, ngroups, headdim, dstate must be >= 1");
  if (a->nheads % a->ngroups != 0)
    return fail(SSD_ERR_INVALID_ARG, "nheads (%lld) is not a multiple of ngroups (%lld)",
                (long long)a->nheads, (long long)a->ngroups);
  if (a->batch > 65535 || a->seqlen >= kMaxDim || a->nheads > 4096)
    return fail(SSD_ERR_UNSUPPORTED, "batch <= 65535, seqlen < 2^31, nheads <= 4096 supported");
  if (a->headdim > 256 || a->dstate > 256)
    return fail(SSD_ERR_UNSUPPORTED, "headdim and dstate up to 256 are supported (got %lld, %lld)",
                (long long)a->headdim, (long long)a->dstate);
  if (a->io_dtype != SSD_DTYPE_F32 && a->io_dtype != SSD_DTYPE_BF16)
    return fail(SSD_ERR_INVALID_ARG, "unknown io_dtype %d", (int)a->io_dtype);
  pr->Q_req = chunk;
  if (chunk == 0) chunk = 64;
  if (chunk != 32 && chunk != 64 && chunk != 128)
    return fail(SSD_ERR_UNSUPPORTED, "chunk size must be 32, 64 or 128 (got %lld)", (long long)chunk);
  int64_t t;
  if (!mul_ok(a->batch, a->seqlen, &t) || !mul_ok(t, a->nheads, &t) || !mul_ok(t, a->headdim, &t) ||
      !mul_ok(a->batch * a->nheads, a->headdim * a->dstate, &t))
    return fail(SSD_ERR_INVALID_ARG, "problem size overflows");
  pr->B = a->batch;
  pr->L = a->seqlen;
  pr->H = a->nheads;
  pr->P = a->headdim;
  pr->G = a->ngroups;
  pr->N = a->dstate;
  pr->io = a->io_dtype;
  pr->Q = chunk;
  pr->nc = (a->seqlen + chunk - 1) / chunk;
  pr->x = a->x;
  pr->dt = a->dt;
  pr->A = a->A;
  pr->Bm = a->Bm;
  pr->Cm = a->Cm;
  pr->D = a->D;
  pr->init = a->init_state;
  pr->y = a->y;
  pr->final_state = a->final_state;
  return SSD_OK;
}

// Pointer checks: presence, alignment, overlap of outputs with inputs.
// `require_y` is false for the step entry points that do not write y.
ssd_status check_pointers(const Problem& p, bool require_y = true) {
  const size_t s = p.io == SSD_DTYPE_BF16 ? 2 : 4;
  const size_t BLH = (size_t)(p.B * p.L * p.H);
  const size_t nx = BLH * p.P * s, ndt = (BLH >> p.rank_log2) * 4, nbc = (size_t)(p.B * p.L * p.G * p.N) * s;
  const size_t nst = (size_t)(p.B * p.H * p.P * p.N) * 4;
  const bool any_tokens = p.B > 0 && p.L > 0;
  if (any_tokens) {
    if (!p.x || !p.dt || !p.A || !p.Bm || !p.Cm || (require_y && !p.y))
      return fail(SSD_ERR_INVALID_ARG, require_y ? "x, dt, A, Bm, Cm and y are required"
                                                 : "x, dt, A, Bm and Cm are required");
  }
  const Span in[] = {{p.x, nx, "x"},          {p.dt, ndt, "dt"},  {p.A, (size_t)p.H * 4, "A"},
                     {p.Bm, nbc, "Bm"},       {p.Cm, nbc, "Cm"},  {p.D, (size_t)p.H * 4, "D"},
                     {p.init, nst, "init_state"}};
  const Span out[] = {{p.y, nx, "y"}, {p.final_state, nst, "final_state"}};
  for (const Span& v : in)
    if (v.p && !aligned16(v.p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v.name);
  for (const Span& v : out)
    if (v.p && !aligned16(v.p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v.name);
  for (const Span& o : out)
    for (const Span& i : in) {
      if (o.p == p.final_state && i.p == p.init && o.p == i.p) continue;  // in-place state
      if (overlaps(o, i)) return fail(SSD_ERR_INVALID_ARG, "%s overlaps input %s", o.name, i.name);
    }
  if (overlaps(out[0], out[1])) return fail(SSD_ERR_INVALID_ARG, "y overlaps final_state");
  return SSD_OK;
}

struct ChunkedWs {
  size_t off_cs, off_dt, off_states, off_bf, total;
};

// The first 256 bytes hold the status word (read by ssd_workspace_status);
// off_bf: bf16 copies of the entering states for the tensor-core chunk
// outputs (only where scan_tc_supported).
ChunkedWs chunked_ws(const Problem& p) {
  ChunkedWs w;
  const size_t ncs = align_up((size_t)(p.B * p.H * p.nc * p.Q) * 4, 256);
  const size_t nst = align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 4, 256);
  const size_t nbf = scan_tc_supported(p) ? align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 2, 256) : 0;
  w.off_cs = 256;
  w.off_dt = w.off_cs + ncs;
  w.off_states = w.off_dt + ncs;
  w.off_bf = w.off_states + nst;
  w.total = w.off_bf + nbf;
  return w;
}

// Which algorithm a call runs.
ssd_status choose_algo(const ssd_fwd_args* a, const Problem& p, int* algo) {
  switch (a->algo) {
    case SSD_ALGO_AUTO:
      *algo = fused_preferred(p) ? SSD_ALGO_FUSED : SSD_ALGO_CHUNKED;
      return SSD_OK;
    case SSD_ALGO_CHUNKED:
      *algo = SSD_ALGO_CHUNKED;
      return SSD_OK;
    case SSD_ALGO_FUSED:
      if (!fused_supported(p))
        return fail(SSD_ERR_UNSUPPORTED,
                    "the fused kernel needs bf16 io, headdim 64, dstate 16, 64 or 128 and chunk 0 or 128");
      *algo = SSD_ALGO_FUSED;
      return SSD_OK;
    default:
      return fail(SSD_ERR_INVALID_ARG, "unknown algo %d", (int)a->algo);
  }
}

// The chunked path's problem: chunk_size 0 is 128 where the tensor-core
// chunk states and outputs apply (bf16, headdim 64, dstate 64 / 128 / 256),
// else 64.
Problem chunked_problem(const Problem& p) {
  if (p.Q_req != 0) return p;
  Problem q = p;
  q.Q = 128;
  q.nc = (q.L + q.Q - 1) / q.Q;
  return scan_tc_supported(q) ? q : p;
}

size_t workspace_for(int algo, const Problem& p) {
  if (p.B == 0 || p.L == 0) return 0;
  return algo == SSD_ALGO_FUSED ? fused_workspace_bytes(p) : chunked_ws(chunked_problem(p)).total;
}

ssd_status finish_launch(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  g_err[0] = '\0';
  return SSD_OK;
}

// Empty sequence: y has no elements; the final state is the initial one.
ssd_status empty_sequence(const Problem& p, cudaStream_t s) {
  if (p.final_state && p.B > 0) {
    const size_t n = (size_t)(p.B * p.H * p.P * p.N) * 4;
    cudaError_t e = p.init ? (p.init == p.final_state
                                  ? cudaSuccess
                                  : cudaMemcpyAsync(p.final_state, p.init, n, cudaMemcpyDeviceToDevice, s))
                           : cudaMemsetAsync(p.final_state, 0, n, s);
    return finish_launch(e, "empty-sequence state copy");
  }
  return finish_launch(cudaSuccess, "");
}

ssd_status step_prologue(const ssd_fwd_args* a, int64_t chunk, Problem* p, bool require_y) {
  ssd_status st = check_shape(a, chunk, p);
  if (st != SSD_OK) return st;
  if (chunk == 0) return fail(SSD_ERR_INVALID_ARG, "the step entry points need an explicit chunk");
  if (p->B == 0 || p->L == 0) return fail(SSD_ERR_INVALID_ARG, "the step entry points need batch, seqlen >= 1");
  return check_pointers(*p, require_y);
}

ssd_status check_buf(const void* q, const char* name) {
  if (!q) return fail(SSD_ERR_INVALID_ARG, "%s is required", name);
  if (!aligned16(q)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

using namespace ssd;

SSD_API int ssd_abi_version(void) { return SSD_ABI_VERSION; }

SSD_API const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "SSD_OK: success";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: invalid argument";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: shape or option not supported";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing or too small";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: CUDA runtime error";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: bounded device wait gave up";
    default: return "unknown ssd_status";
  }
}

SSD_API const char* ssd_last_error_message(void) { return g_err; }

SSD_API ssd_status ssd_workspace_status(const void* workspace, void* stream) {
  if (!workspace) return fail(SSD_ERR_INVALID_ARG, "workspace is NULL");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the workspace status");
  if (word == (int32_t)SSD_ERR_TIMEOUT) return fail(SSD_ERR_TIMEOUT, "a bounded device-side wait gave up");
  g_err[0] = '\0';
  return SSD_OK;
}

SSD_API size_t ssd_fwd_workspace_size(const ssd_fwd_args* a) {
  Problem p;
  if (check_shape(a, a ? a->chunk_size : 0, &p) != SSD_OK) return (size_t)-1;
  int algo = 0;
  if (choose_algo(a, p, &algo) != SSD_OK) return (size_t)-1;
  return workspace_for(algo, p);
}

namespace ssd {
namespace {
ssd_status run_chunked(const Problem& p, void* workspace, cudaStream_t s);

// ssd_fwd and ssd_fwd_ex after their own checks: choose the path, check the
// workspace, launch.
ssd_status run_fwd(const ssd_fwd_args* a, const Problem& p, void* stream) {
  ssd_status st;
  int algo = 0;
  if ((st = choose_algo(a, p, &algo)) != SSD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0) return finish_launch(cudaSuccess, "");
  if (p.L == 0) return empty_sequence(p, s);
  const size_t need = workspace_for(algo, p);
  if (need > 0 && (!a->workspace || a->workspace_bytes < need))
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                a->workspace ? a->workspace_bytes : (size_t)0);
  if (need > 0 && (reinterpret_cast<uintptr_t>(a->workspace) & 255u))
    return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  if (need > 0) {
    const Span ws{a->workspace, need, "workspace"};
    const size_t sio = p.io == SSD_DTYPE_BF16 ? 2 : 4;
    const Span others[] = {{p.x, (size_t)(p.B * p.L * p.H * p.P) * sio, "x"},
                           {p.y, (size_t)(p.B * p.L * p.H * p.P) * sio, "y"},
                           {p.final_state, (size_t)(p.B * p.H * p.P * p.N) * 4, "final_state"},
                           {p.init, (size_t)(p.B * p.H * p.P * p.N) * 4, "init_state"},
                           {p.z, (size_t)(p.B * p.L * p.H * p.P) * sio, "z"}};
    for (const Span& o : others)
      if (overlaps(ws, o)) return fail(SSD_ERR_INVALID_ARG, "workspace overlaps %s", o.name);
  }
  if (algo == SSD_ALGO_FUSED) return finish_launch(launch_fused(p, a->workspace, s), "fused kernel");
  return run_chunked(chunked_problem(p), a->workspace, s);
}

ssd_status run_chunked(const Problem& pin, void* workspace, cudaStream_t s) {
  const ChunkedWs w = chunked_ws(pin);
  char* base = static_cast<char*>(workspace);
  Problem p = pin;
  p.err = reinterpret_cast<int32_t*>(base);  // status word, cleared on every call
  float* dA_cs = reinterpret_cast<float*>(base + w.off_cs);
  float* dt_c = reinterpret_cast<float*>(base + w.off_dt);
  float* states = reinterpret_cast<float*>(base + w.off_states);
  cudaError_t e = cudaMemsetAsync(p.err, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "status word");
  e = launch_chunk_cumsum(p, dA_cs, dt_c, s);
  if (e != cudaSuccess) return cuda_fail(e, "chunk_cumsum");
  if ((e = launch_chunk_state(p, dA_cs, dt_c, states, s)) != cudaSuccess) return cuda_fail(e, "chunk_state");
  if (w.off_bf != w.total) {  // tensor-core chunk outputs from bf16 entering states
    void* st_bf = base + w.off_bf;
    if ((e = launch_state_passing(p, dA_cs, states, s, st_bf)) != cudaSuccess) return cuda_fail(e, "state_passing");
    return finish_launch(launch_chunk_scan_tc(p, dA_cs, dt_c, nullptr, st_bf, nullptr, s), "chunk_scan");
  }
  if ((e = launch_state_passing(p, dA_cs, states, s)) != cudaSuccess) return cuda_fail(e, "state_passing");
  return finish_launch(launch_chunk_scan(p, dA_cs, dt_c, states, s), "chunk_scan");
}
}  // namespace
}  // namespace ssd

SSD_API ssd_status ssd_fwd(const ssd_fwd_args* a, void* stream) {
  Problem p;
  ssd_status st = check_shape(a, a ? a->chunk_size : 0, &p);
  if (st != SSD_OK) return st;
  if ((st = check_pointers(p)) != SSD_OK) return st;
  return run_fwd(a, p, stream);
}

namespace ssd {
namespace {
// Pipelining of ssd_fwd_host.  The problem is cut into groups of `rows`
// batch rows by `nt` tokens; a group's inputs are copied in while the
// previous group is computed and the one before it copied out.  Sequences of
// at least four 128-token chunks are cut along the tokens (all rows in every
// group, up to 16 token segments of whole 128-token chunks, the state handed
// from one segment to the next in a device buffer), shorter ones along the
// batch rows (four row groups).  Device layout: a 256-byte status word, two
// staging slots (inputs, y, the forward pass's workspace), two pairs of state
// buffers (a pair per row group, alternating between row groups; a segment
// reads one buffer of its pair and writes the other), then A and D.
struct HostPlan {
  int64_t rows, row_groups, nt, segs;
  size_t ws;  // forward-pass workspace of the largest group
  size_t off_x, off_dt, off_b, off_c, off_y, off_ws, slot, off_slots, st, off_carry, off_A, off_D, total;
};

HostPlan host_plan(const ssd_fwd_args* a, const Problem& p, int algo) {
  (void)a;
  HostPlan h;
  const int64_t nc128 = (p.L + 127) / 128;
  if (nc128 >= 4) {
    h.rows = p.B;
    h.segs = std::min<int64_t>(16, nc128);
    h.nt = (nc128 + h.segs - 1) / h.segs * 128;
    h.segs = (p.L + h.nt - 1) / h.nt;
  } else {
    h.rows = std::max<int64_t>(1, (p.B + 3) / 4);
    h.segs = 1;
    h.nt = p.L;
  }
  h.row_groups = (p.B + h.rows - 1) / h.rows;
  const size_t sio = p.io == SSD_DTYPE_BF16 ? 2 : 4;
  // workspace of the largest of the group shapes (full and last rows, full and last segment)
  h.ws = 0;
  for (const int64_t nb : {h.rows, p.B % h.rows}) {
    for (const int64_t nl : {h.nt, p.L - (h.segs - 1) * h.nt}) {
      if (nb <= 0 || nl <= 0) continue;
      Problem g = p;
      g.B = nb;
      g.L = nl;
      g.nc = (g.L + g.Q - 1) / g.Q;
      h.ws = std::max(h.ws, workspace_for(algo, g));
    }
  }
  size_t o = 0;
  auto take = [&](size_t n) {
    const size_t at = o;
    o += align_up(n, 256);
    return at;
  };
  const size_t tok = (size_t)(h.rows * h.nt);
  h.off_x = take(tok * p.H * p.P * sio);
  h.off_dt = take(tok * p.H * 4);
  h.off_b = take(tok * p.G * p.N * sio);
  h.off_c = take(tok * p.G * p.N * sio);
  h.off_y = take(tok * p.H * p.P * sio);
  h.off_ws = take(h.ws);
  h.slot = o;
  h.off_slots = 256;
  h.st = (size_t)(h.rows * p.H * p.P * p.N) * 4;
  h.off_carry = h.off_slots + 2 * h.slot;
  h.off_A = h.off_carry + 4 * align_up(h.st, 256);
  h.off_D = h.off_A + align_up((size_t)p.H * 4, 256);
  h.total = h.off_D + align_up((size_t)p.H * 4, 256);
  return h;
}
}  // namespace
}  // namespace ssd

namespace ssd {
namespace {
// The copy streams and events of ssd_fwd_host, created once per device and
// kept until the process exits.  Calls on one device hold its mutex while
// they enqueue (the events are re-recorded by every call).
struct HostStreams {
  std::mutex mu;
  bool ready = false;
  cudaStream_t s_in = nullptr, s_out = nullptr;
  cudaEvent_t ev[9] = {};  // entry, in[2], comp[2], out[2], state out[2]
};

HostStreams* host_streams(int dev) {
  constexpr int kMaxDevices = 64;
  static HostStreams all[kMaxDevices];
  return dev >= 0 && dev < kMaxDevices ? &all[dev] : nullptr;
}

// Keeps the first non-zero status of a group's forward pass in the call's word.
__global__ void status_merge_kernel(int32_t* dst, const int32_t* src) {
  if (threadIdx.x == 0 && *src != 0 && *dst == 0) *dst = *src;
}
}  // namespace
}  // namespace ssd

SSD_API size_t ssd_fwd_host_workspace_size(const ssd_fwd_args* a) {
  Problem p;
  if (check_shape(a, a ? a->chunk_size : 0, &p) != SSD_OK) return (size_t)-1;
  int algo = 0;
  if (choose_algo(a, p, &algo) != SSD_OK) return (size_t)-1;
  if (p.B == 0 || p.L == 0) return 0;
  return host_plan(a, p, algo).total;
}

SSD_API ssd_status ssd_fwd_host(const ssd_fwd_args* a, void* stream) {
  Problem p;
  ssd_status st = check_shape(a, a ? a->chunk_size : 0, &p);
  if (st != SSD_OK) return st;
  int algo = 0;
  if ((st = choose_algo(a, p, &algo)) != SSD_OK) return st;
  if (p.B == 0) return finish_launch(cudaSuccess, "");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t sio = p.io == SSD_DTYPE_BF16 ? 2 : 4;
  if (p.L == 0) {  // no tokens: the final state is the initial one
    if (!a->final_state) return finish_launch(cudaSuccess, "");
    const size_t n = (size_t)(p.B * p.H * p.P * p.N) * 4;
    if (a->init_state) return finish_launch(cudaMemcpyAsync(a->final_state, a->init_state, n, cudaMemcpyHostToHost, s),
                                            "host copy");
    std::memset(a->final_state, 0, n);
    return finish_launch(cudaSuccess, "");
  }
  if (!a->x || !a->dt || !a->A || !a->Bm || !a->Cm || !a->y)
    return fail(SSD_ERR_INVALID_ARG, "x, dt, A, Bm, Cm and y are required");
  const HostPlan h = host_plan(a, p, algo);
  if (!a->workspace || a->workspace_bytes < h.total)
    return fail(SSD_ERR_WORKSPACE, "device workspace of %zu bytes needed, %zu given", h.total,
                a->workspace ? a->workspace_bytes : (size_t)0);
  if (reinterpret_cast<uintptr_t>(a->workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  char* dev = static_cast<char*>(a->workspace);
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  HostStreams* hs = host_streams(device);
  if (!hs) return fail(SSD_ERR_UNSUPPORTED, "device ordinal %d out of range", device);
  std::lock_guard<std::mutex> lock(hs->mu);
  if (!hs->ready) {
    e = cudaStreamCreateWithFlags(&hs->s_in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hs->s_out, cudaStreamNonBlocking);
    for (int i = 0; i < 9 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&hs->ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "ssd_fwd_host streams");
    hs->ready = true;
  }
  cudaStream_t s_in = hs->s_in, s_out = hs->s_out;
  cudaEvent_t ev_entry = hs->ev[0], *ev_in = hs->ev + 1, *ev_comp = hs->ev + 3, *ev_out = hs->ev + 5,
              *ev_st = hs->ev + 7;
  int32_t* status = reinterpret_cast<int32_t*>(dev);  // the call's status word
  e = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
  // everything below is ordered after the work already on `stream`
  if (e == cudaSuccess) e = cudaEventRecord(ev_entry, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_in, ev_entry, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_entry, 0);
  float* dA = reinterpret_cast<float*>(dev + h.off_A);
  float* dD = a->D ? reinterpret_cast<float*>(dev + h.off_D) : nullptr;
  if (e == cudaSuccess) e = cudaMemcpyAsync(dA, a->A, (size_t)p.H * 4, cudaMemcpyHostToDevice, s_in);
  if (e == cudaSuccess && dD) e = cudaMemcpyAsync(dD, a->D, (size_t)p.H * 4, cudaMemcpyHostToDevice, s_in);
  // bytes per token of each tensor (a batch row of the host tensors is L of them)
  const size_t tx = (size_t)(p.H * p.P) * sio, tdt = (size_t)p.H * 4, tbc = (size_t)(p.G * p.N) * sio;
  auto hp = [](const void* q, size_t off) { return static_cast<const char*>(q) + off; };
  ssd_status result = SSD_OK;
  int64_t gi = 0;
  for (int64_t r = 0; r < h.row_groups && e == cudaSuccess && result == SSD_OK; ++r) {
    const int64_t b0 = r * h.rows, nb = std::min(h.rows, p.B - b0);
    const int cs = (int)(r & 1);  // state buffer pair of this row group
    float* carry[2];
    for (int q = 0; q < 2; ++q)
      carry[q] = reinterpret_cast<float*>(dev + h.off_carry + (2 * cs + q) * align_up(h.st, 256));
    const size_t fst = (size_t)(nb * p.H * p.P * p.N) * 4, ost = (size_t)(b0 * p.H * p.P * p.N) * 4;
    // the row group's initial state into its buffer, once the buffer's last
    // final state (two row groups back) has been copied out
    if (r >= 2) e = cudaStreamWaitEvent(s_in, ev_st[cs], 0);
    if (e == cudaSuccess && a->init_state)
      e = cudaMemcpyAsync(carry[0], hp(a->init_state, ost), fst, cudaMemcpyHostToDevice, s_in);
    for (int64_t j = 0; j < h.segs && e == cudaSuccess && result == SSD_OK; ++j, ++gi) {
      const int sl = (int)(gi & 1);
      const int64_t t0 = j * h.nt, nl = std::min(h.nt, p.L - t0);
      char* slot = dev + h.off_slots + sl * h.slot;
      // host offset of (row b0, token t0) for a tensor of `t` bytes per token
      auto off = [&](size_t t) { return ((size_t)b0 * p.L + t0) * t; };
      auto in2d = [&](size_t dst_off, const void* src, size_t t) {
        return cudaMemcpy2DAsync(slot + dst_off, nl * t, hp(src, off(t)), p.L * t, nl * t, nb,
                                 cudaMemcpyHostToDevice, s_in);
      };
      // copies in, once the slot's previous outputs have been copied out
      if (gi >= 2) e = cudaStreamWaitEvent(s_in, ev_out[sl], 0);
      if (e == cudaSuccess) e = in2d(h.off_x, a->x, tx);
      if (e == cudaSuccess) e = in2d(h.off_dt, a->dt, tdt);
      if (e == cudaSuccess) e = in2d(h.off_b, a->Bm, tbc);
      if (e == cudaSuccess) e = in2d(h.off_c, a->Cm, tbc);
      if (e == cudaSuccess) e = cudaEventRecord(ev_in[sl], s_in);
      // the forward pass of the group on `stream`: segment j's state enters
      // from buffer j % 2 of the pair (the initial state, or segment j-1's
      // final state) and leaves into the other one
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev_in[sl], 0);
      if (e != cudaSuccess) break;
      ssd_fwd_args g = *a;
      g.batch = nb;
      g.seqlen = nl;
      g.x = slot + h.off_x;
      g.dt = reinterpret_cast<const float*>(slot + h.off_dt);
      g.A = dA;
      g.Bm = slot + h.off_b;
      g.Cm = slot + h.off_c;
      g.D = dD;
      g.init_state = (j > 0 || a->init_state) ? carry[j & 1] : nullptr;
      g.y = slot + h.off_y;
      g.final_state = carry[(j + 1) & 1];
      g.workspace = slot + h.off_ws;
      g.workspace_bytes = h.ws;
      Problem pg;
      if ((result = check_shape(&g, g.chunk_size, &pg)) != SSD_OK) break;
      if ((result = run_fwd(&g, pg, stream)) != SSD_OK) break;
      status_merge_kernel<<<1, 32, 0, s>>>(status, reinterpret_cast<const int32_t*>(slot + h.off_ws));
      if ((e = cudaGetLastError()) != cudaSuccess) break;
      e = cudaEventRecord(ev_comp[sl], s);
      // copies out: y of the group, and after the row group's last segment its final state
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s_out, ev_comp[sl], 0);
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(static_cast<char*>(a->y) + off(tx), p.L * tx, slot + h.off_y, nl * tx, nl * tx, nb,
                              cudaMemcpyDeviceToHost, s_out);
      if (e == cudaSuccess) e = cudaEventRecord(ev_out[sl], s_out);
      if (e == cudaSuccess && j == h.segs - 1) {
        if (a->final_state)
          e = cudaMemcpyAsync(reinterpret_cast<char*>(a->final_state) + ost, carry[(j + 1) & 1], fst,
                              cudaMemcpyDeviceToHost, s_out);
        if (e == cudaSuccess) e = cudaEventRecord(ev_st[cs], s_out);
      }
    }
  }
  // `stream` completes after the last copies out
  for (int sl = 0; sl < 2 && e == cudaSuccess; ++sl)
    if (gi > sl) e = cudaStreamWaitEvent(s, ev_out[sl], 0);
  for (int c = 0; c < 2 && e == cudaSuccess; ++c)
    if (h.row_groups > c) e = cudaStreamWaitEvent(s, ev_st[c], 0);
  if (result != SSD_OK) return result;
  return finish_launch(e, "ssd_fwd_host");
}

SSD_API size_t ssd_fwd_ex_workspace_size(const ssd_fwd_ex_args* a) {
  return a ? ssd_fwd_workspace_size(&a->base) : (size_t)-1;
}

SSD_API ssd_status ssd_fwd_ex(const ssd_fwd_ex_args* a, void* stream) {
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  Problem p;
  ssd_status st = check_shape(&a->base, a->base.chunk_size, &p);
  if (st != SSD_OK) return st;
  if ((st = check_pointers(p)) != SSD_OK) return st;
  if (a->reserved != 0) return fail(SSD_ERR_INVALID_ARG, "reserved must be 0");
  if (a->dt_softplus != 0 && a->dt_softplus != 1) return fail(SSD_ERR_INVALID_ARG, "dt_softplus must be 0 or 1");
  const size_t sio = p.io == SSD_DTYPE_BF16 ? 2 : 4;
  const Span zs{a->z, (size_t)(p.B * p.L * p.H * p.P) * sio, "z"};
  const Span bs{a->dt_bias, (size_t)p.H * 4, "dt_bias"};
  for (const Span* v : {&zs, &bs})
    if (v->p && !aligned16(v->p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v->name);
  const Span outs[] = {{p.y, (size_t)(p.B * p.L * p.H * p.P) * sio, "y"},
                       {p.final_state, (size_t)(p.B * p.H * p.P * p.N) * 4, "final_state"}};
  for (const Span& o : outs)
    for (const Span* v : {&zs, &bs})
      if (overlaps(o, *v)) return fail(SSD_ERR_INVALID_ARG, "%s overlaps input %s", o.name, v->name);
  p.dt_bias = a->dt_bias;
  p.dt_softplus = a->dt_softplus;
  p.z = a->z;
  return run_fwd(&a->base, p, stream);
}

// Allocation-free variant of ssd_fwd: the fused kernel with its workspace in
// the library's fixed device array instead of caller memory.
SSD_API ssd_status ssd_fwd_noalloc(const ssd_fwd_args* a, void* stream) {
  Problem p;
  ssd_status st = check_shape(a, a ? a->chunk_size : 0, &p);
  if (st != SSD_OK) return st;
  if ((st = check_pointers(p)) != SSD_OK) return st;
  if (a->algo != SSD_ALGO_AUTO && a->algo != SSD_ALGO_FUSED)
    return fail(SSD_ERR_UNSUPPORTED, "ssd_fwd_noalloc runs the fused kernel only (algo auto or fused)");
  if (!fused_supported(p))
    return fail(SSD_ERR_UNSUPPORTED,
                "ssd_fwd_noalloc needs the fused kernel: bf16 io, headdim 64, dstate 16, 64 or 128, chunk 0 or 128");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0) return finish_launch(cudaSuccess, "");
  if (p.L == 0) return empty_sequence(p, s);
  const size_t need = fused_workspace_bytes(p, static_scratch_bytes());
  if (need > static_scratch_bytes())
    return fail(SSD_ERR_UNSUPPORTED, "ssd_fwd_noalloc: this problem needs %zu bytes of scratch, the fixed "
                "scratch holds %zu", need, static_scratch_bytes());
  void* scratch = nullptr;
  cudaError_t e = static_scratch_ptr(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
  return finish_launch(launch_fused(p, scratch, s, static_scratch_bytes()), "fused kernel (no-alloc)");
}

namespace ssd {
namespace {
// ssd_fwd_mimo's problem: the rows (token, rank) as the sequence of the fused kernel.
ssd_status mimo_problem(const ssd_fwd_mimo_args* a, Problem* p) {
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  const int64_t R = a->rank;
  if (R != 1 && R != 2 && R != 4 && R != 8) return fail(SSD_ERR_UNSUPPORTED, "rank must be 1, 2, 4 or 8");
  if (a->base.seqlen < 0 || a->base.seqlen > (int64_t(1) << 27))
    return fail(SSD_ERR_INVALID_ARG, "seqlen must be in [0, 2^27]");
  ssd_fwd_args rows = a->base;
  rows.seqlen = a->base.seqlen * R;
  ssd_status st = check_shape(&rows, rows.chunk_size, p);
  if (st != SSD_OK) return st;
  p->rank_log2 = R == 1 ? 0 : R == 2 ? 1 : R == 4 ? 2 : 3;
  if ((st = check_pointers(*p)) != SSD_OK) return st;
  if (a->base.algo != SSD_ALGO_AUTO && a->base.algo != SSD_ALGO_FUSED)
    return fail(SSD_ERR_UNSUPPORTED, "ssd_fwd_mimo runs the fused kernel only (algo auto or fused)");
  if (!fused_supported(*p))
    return fail(SSD_ERR_UNSUPPORTED,
                "ssd_fwd_mimo needs the fused kernel: bf16 io, headdim 64, dstate 16, 64, 128 or 256, chunk 0 or 128");
  return SSD_OK;
}
}  // namespace
}  // namespace ssd

SSD_API size_t ssd_fwd_mimo_workspace_size(const ssd_fwd_mimo_args* a) {
  Problem p;
  if (mimo_problem(a, &p) != SSD_OK) return (size_t)-1;
  if (p.B == 0 || p.L == 0) return 0;
  return fused_workspace_bytes(p);
}

SSD_API ssd_status ssd_fwd_mimo(const ssd_fwd_mimo_args* a, void* stream) {
  Problem p;
  ssd_status st = mimo_problem(a, &p);
  if (st != SSD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0) return finish_launch(cudaSuccess, "");
  if (p.L == 0) return empty_sequence(p, s);
  const size_t need = fused_workspace_bytes(p);
  if (!a->base.workspace || a->base.workspace_bytes < need)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                a->base.workspace ? a->base.workspace_bytes : (size_t)0);
  if (reinterpret_cast<uintptr_t>(a->base.workspace) & 255u)
    return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
  const size_t sio = 2;
  const Span ws{a->base.workspace, need, "workspace"};
  const Span others[] = {{p.x, (size_t)(p.B * p.L * p.H * p.P) * sio, "x"},
                         {p.y, (size_t)(p.B * p.L * p.H * p.P) * sio, "y"},
                         {p.final_state, (size_t)(p.B * p.H * p.P * p.N) * 4, "final_state"},
                         {p.init, (size_t)(p.B * p.H * p.P * p.N) * 4, "init_state"}};
  for (const Span& o : others)
    if (overlaps(ws, o)) return fail(SSD_ERR_INVALID_ARG, "workspace overlaps %s", o.name);
  return finish_launch(launch_fused(p, a->base.workspace, s), "fused kernel (retrieval rank)");
}

SSD_API ssd_status ssd_fwd_noalloc_status(void* stream) {
  void* scratch = nullptr;
  cudaError_t e = static_scratch_ptr(&scratch);
  if (e != cudaSuccess) return cuda_fail(e, "static scratch address");
  return ssd_workspace_status(scratch, stream);
}

SSD_API ssd_status ssd_step(const ssd_step_args* a, void* stream) {
  using namespace ssd;
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  if (a->batch < 0) return fail(SSD_ERR_INVALID_ARG, "batch must be >= 0");
  if (a->nheads < 1 || a->ngroups < 1 || a->headdim < 1 || a->dstate < 1)
    return fail(SSD_ERR_INVALID_ARG, "nheads, ngroups, headdim, dstate must be >= 1");
  if (a->nheads % a->ngroups != 0)
    return fail(SSD_ERR_INVALID_ARG, "nheads (%lld) is not a multiple of ngroups (%lld)",
                (long long)a->nheads, (long long)a->ngroups);
  if (a->headdim > 256 || a->dstate > 256)
    return fail(SSD_ERR_UNSUPPORTED, "headdim and dstate up to 256 are supported (got %lld, %lld)",
                (long long)a->headdim, (long long)a->dstate);
  if (a->batch > 65535 || a->nheads > 4096)
    return fail(SSD_ERR_UNSUPPORTED, "batch <= 65535 and nheads <= 4096 supported");
  if (a->io_dtype != SSD_DTYPE_F32 && a->io_dtype != SSD_DTYPE_BF16)
    return fail(SSD_ERR_INVALID_ARG, "unknown io_dtype %d", (int)a->io_dtype);
  if (a->reserved != 0) return fail(SSD_ERR_INVALID_ARG, "reserved must be 0");
  if (a->batch == 0) return SSD_OK;
  if (!a->x || !a->dt || !a->A || !a->Bm || !a->Cm || !a->state || !a->y)
    return fail(SSD_ERR_INVALID_ARG, "x, dt, A, Bm, Cm, state and y must not be NULL");
  const void* ptrs[] = {a->x, a->dt, a->A, a->Bm, a->Cm, a->D, a->state, a->y};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return fail(SSD_ERR_INVALID_ARG, "every pointer must be 16-byte aligned");
  const size_t io = a->io_dtype == SSD_DTYPE_BF16 ? 2 : 4;
  const size_t B = (size_t)a->batch, H = (size_t)a->nheads, P = (size_t)a->headdim, G = (size_t)a->ngroups,
               N = (size_t)a->dstate;
  const Span in[] = {{a->x, B * H * P * io, "x"},     {a->dt, B * H * 4, "dt"},
                     {a->A, H * 4, "A"},               {a->Bm, B * G * N * io, "Bm"},
                     {a->Cm, B * G * N * io, "Cm"},    {a->D, a->D ? H * 4 : 0, "D"}};
  const Span y{a->y, B * H * P * io, "y"}, st{a->state, B * H * P * N * 4, "state"};
  for (const Span& s : in) {
    if (overlaps(y, s)) return fail(SSD_ERR_INVALID_ARG, "y overlaps %s", s.name);
    if (overlaps(st, s)) return fail(SSD_ERR_INVALID_ARG, "state overlaps %s", s.name);
  }
  if (overlaps(y, st)) return fail(SSD_ERR_INVALID_ARG, "y overlaps state");
  StepProblem q;
  q.B = a->batch;
  q.H = a->nheads;
  q.P = a->headdim;
  q.G = a->ngroups;
  q.N = a->dstate;
  q.io = a->io_dtype;
  q.x = a->x;
  q.dt = a->dt;
  q.A = a->A;
  q.Bm = a->Bm;
  q.Cm = a->Cm;
  q.D = a->D;
  q.state = a->state;
  q.y = a->y;
  const cudaError_t e = launch_step(q, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "ssd_step launch");
  return SSD_OK;
}

SSD_API ssd_status ssd_chunk_cumsum(const ssd_fwd_args* a, int64_t chunk, float* dA_cs,
                                    float* dt_chunked, void* stream) {
  Problem p;
  ssd_status st = step_prologue(a, chunk, &p, false);
  if (st != SSD_OK) return st;
  if ((st = check_buf(dA_cs, "dA_cs")) != SSD_OK || (st = check_buf(dt_chunked, "dt_chunked")) != SSD_OK)
    return st;
  return finish_launch(launch_chunk_cumsum(p, dA_cs, dt_chunked, reinterpret_cast<cudaStream_t>(stream)),
                       "chunk_cumsum");
}

SSD_API ssd_status ssd_chunk_state(const ssd_fwd_args* a, int64_t chunk, const float* dA_cs,
                                   const float* dt_chunked, float* states, void* stream) {
  Problem p;
  ssd_status st = step_prologue(a, chunk, &p, false);
  if (st != SSD_OK) return st;
  if ((st = check_buf(dA_cs, "dA_cs")) != SSD_OK || (st = check_buf(dt_chunked, "dt_chunked")) != SSD_OK ||
      (st = check_buf(states, "states")) != SSD_OK)
    return st;
  return finish_launch(
      launch_chunk_state(p, dA_cs, dt_chunked, states, reinterpret_cast<cudaStream_t>(stream)),
      "chunk_state");
}

SSD_API ssd_status ssd_state_passing(const ssd_fwd_args* a, int64_t chunk, const float* dA_cs,
                                     float* states, void* stream) {
  Problem p;
  ssd_status st = step_prologue(a, chunk, &p, false);
  if (st != SSD_OK) return st;
  if ((st = check_buf(dA_cs, "dA_cs")) != SSD_OK || (st = check_buf(states, "states")) != SSD_OK) return st;
  return finish_launch(launch_state_passing(p, dA_cs, states, reinterpret_cast<cudaStream_t>(stream)),
                       "state_passing");
}

SSD_API ssd_status ssd_chunk_scan(const ssd_fwd_args* a, int64_t chunk, const float* dA_cs,
                                  const float* dt_chunked, const float* states, void* stream) {
  Problem p;
  ssd_status st = step_prologue(a, chunk, &p, true);
  if (st != SSD_OK) return st;
  if ((st = check_buf(dA_cs, "dA_cs")) != SSD_OK || (st = check_buf(dt_chunked, "dt_chunked")) != SSD_OK ||
      (st = check_buf(states, "states")) != SSD_OK)
    return st;
  return finish_launch(
      launch_chunk_scan(p, dA_cs, dt_chunked, states, reinterpret_cast<cudaStream_t>(stream)),
      "chunk_scan");
}

// ---------------------------------------------------------------- backward pass
namespace ssd {
namespace {

ssd_status bwd_prologue(const ssd_bwd_args* a, BwdProblem* q) {
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  ssd_status st = check_shape(&a->fwd, a->fwd.chunk_size, &q->fwd);
  if (st != SSD_OK) return st;
  Problem& p = q->fwd;
  const int qb = bwd_chunk(p, a->fwd.chunk_size);
  if (qb == 0)
    return fail(SSD_ERR_UNSUPPORTED,
                "the backward pass takes chunk 64, or 128 with bf16, headdim 64, dstate 128 (got %lld)",
                (long long)a->fwd.chunk_size);
  p.Q = qb;
  p.nc = (p.L + p.Q - 1) / p.Q;
  if (p.P > bwd_max_headdim())
    return fail(SSD_ERR_UNSUPPORTED, "the backward pass supports headdim up to %d (got %lld)", bwd_max_headdim(),
                (long long)p.P);
  p.y = nullptr;
  p.final_state = nullptr;
  q->dy = a->dy;
  q->dfinal = a->dfinal;
  q->dx = a->dx;
  q->ddt = a->ddt;
  q->dA = a->dA;
  q->dBm = a->dBm;
  q->dCm = a->dCm;
  q->dD = a->dD;
  q->dinit = a->dinit;
  if ((st = check_pointers(p, false)) != SSD_OK) return st;
  const bool tokens = p.B > 0 && p.L > 0;
  if (!q->dA) return fail(SSD_ERR_INVALID_ARG, "dA is required");
  if (tokens && (!q->dy || !q->dx || !q->ddt || !q->dBm || !q->dCm))
    return fail(SSD_ERR_INVALID_ARG, "dy, dx, ddt, dBm and dCm are required");
  const size_t s = p.io == SSD_DTYPE_BF16 ? 2 : 4;
  const size_t BLH = (size_t)(p.B * p.L * p.H);
  const size_t nx = BLH * p.P * s, ndt = BLH * 4, nbc = (size_t)(p.B * p.L * p.G * p.N) * s;
  const size_t nst = (size_t)(p.B * p.H * p.P * p.N) * 4, nh = (size_t)p.H * 4;
  const Span in[] = {{p.x, nx, "x"},   {p.dt, ndt, "dt"},         {p.A, nh, "A"},
                     {p.Bm, nbc, "Bm"}, {p.Cm, nbc, "Cm"},        {p.D, nh, "D"},
                     {p.init, nst, "init_state"}, {q->dy, nx, "dy"}, {q->dfinal, nst, "dfinal"}};
  const Span out[] = {{q->dx, nx, "dx"},   {q->ddt, ndt, "ddt"}, {q->dA, nh, "dA"},      {q->dBm, nbc, "dBm"},
                      {q->dCm, nbc, "dCm"}, {q->dD, nh, "dD"},    {q->dinit, nst, "dinit"}};
  for (const Span& v : in)
    if (v.p && !aligned16(v.p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v.name);
  for (const Span& v : out)
    if (v.p && !aligned16(v.p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v.name);
  for (size_t i = 0; i < sizeof(out) / sizeof(out[0]); ++i) {
    for (const Span& v : in)
      if (overlaps(out[i], v)) return fail(SSD_ERR_INVALID_ARG, "%s overlaps input %s", out[i].name, v.name);
    for (size_t j = i + 1; j < sizeof(out) / sizeof(out[0]); ++j)
      if (overlaps(out[i], out[j])) return fail(SSD_ERR_INVALID_ARG, "%s overlaps %s", out[i].name, out[j].name);
  }
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

SSD_API size_t ssd_bwd_workspace_size(const ssd_bwd_args* a) {
  BwdProblem q;
  if (!a) return (size_t)-1;
  if (check_shape(&a->fwd, a->fwd.chunk_size, &q.fwd) != SSD_OK) return (size_t)-1;
  const int qb = bwd_chunk(q.fwd, a->fwd.chunk_size);
  if (qb == 0) return (size_t)-1;
  if (q.fwd.P > bwd_max_headdim()) return (size_t)-1;
  if (q.fwd.B == 0 || q.fwd.L == 0) return 0;
  q.fwd.Q = qb;
  q.fwd.nc = (q.fwd.L + q.fwd.Q - 1) / q.fwd.Q;
  return bwd_ws(q.fwd).total;
}

SSD_API ssd_status ssd_bwd(const ssd_bwd_args* a, void* stream) {
  BwdProblem q;
  ssd_status st = bwd_prologue(a, &q);
  if (st != SSD_OK) return st;
  const Problem& p = q.fwd;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0 || p.L == 0) {
    // no tokens: final_state = init_state, so dinit = dfinal; dA = dD = 0
    cudaError_t e = cudaMemsetAsync(q.dA, 0, (size_t)p.H * 4, s);
    if (e == cudaSuccess && q.dD) e = cudaMemsetAsync(q.dD, 0, (size_t)p.H * 4, s);
    if (e == cudaSuccess && q.dinit && p.B > 0) {
      const size_t n = (size_t)(p.B * p.H * p.P * p.N) * 4;
      e = q.dfinal ? cudaMemcpyAsync(q.dinit, q.dfinal, n, cudaMemcpyDeviceToDevice, s)
                   : cudaMemsetAsync(q.dinit, 0, n, s);
    }
    return finish_launch(e, "empty backward");
  }
  const size_t need = bwd_ws(p).total;
  if (!a->fwd.workspace || a->fwd.workspace_bytes < need)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                a->fwd.workspace ? a->fwd.workspace_bytes : (size_t)0);
  if (!aligned16(a->fwd.workspace)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  return finish_launch(launch_bwd(q, a->fwd.workspace, s), "backward pass");
}

// ---------------------------------------------------------------- complex decay
namespace ssd {
namespace {

struct RotWs {
  size_t off_cs, off_dt, off_phi, off_re, off_im, off_bf, nbf, total;
};

// off_bf: bf16 copies of the real and imaginary entering states (nbf bytes
// each) for the tensor-core chunk outputs, only where scan_tc_supported.
RotWs rot_ws(const Problem& p) {
  RotWs w;
  const size_t ncs = align_up((size_t)(p.B * p.H * p.nc * p.Q) * 4, 256);
  const size_t nst = align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 4, 256);
  w.nbf = scan_tc_supported(p) ? align_up((size_t)(p.B * p.nc * p.H * p.P * p.N) * 2, 256) : 0;
  w.off_cs = 256;  // the first 256 bytes hold the status word
  w.off_dt = w.off_cs + ncs;
  w.off_phi = w.off_dt + ncs;
  w.off_re = w.off_phi + ncs;
  w.off_im = w.off_re + nst;
  w.off_bf = w.off_im + nst;
  w.total = w.off_bf + 2 * w.nbf;
  return w;
}

// Chunk length of the complex-decay pass: chunk_size 0 is 128 where the
// tensor-core chunk outputs apply, else 64.
void rot_default_chunk(const ssd_fwd_rot_args* a, Problem* p) {
  if (a->base.chunk_size != 0) return;
  Problem q = *p;
  q.Q = 128;
  q.nc = (q.L + q.Q - 1) / q.Q;
  if (scan_tc_supported(q)) *p = q;
}

// The complex decay on the fused kernel (state on chip): bf16 io, headdim 64,
// dstate 128, chunk 0 or 128, algo auto or fused.  Otherwise the chunked path.
bool rot_fused(const ssd_fwd_rot_args* a, const Problem& p) {
  return (a->base.algo == SSD_ALGO_AUTO || a->base.algo == SSD_ALGO_FUSED) && p.N == 128 &&
         (a->base.chunk_size == 0 || a->base.chunk_size == 128) && fused_supported(p);
}

ssd_status rot_prologue(const ssd_fwd_rot_args* a, Problem* p) {
  if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
  ssd_status st = check_shape(&a->base, a->base.chunk_size, p);
  if (st != SSD_OK) return st;
  rot_default_chunk(a, p);
  p->theta = a->theta;
  p->init_im = a->init_state_im;
  p->final_im = a->final_state_im;
  p->complex_decay = true;
  if ((st = check_pointers(*p)) != SSD_OK) return st;
  const bool tokens = p->B > 0 && p->L > 0;
  if (tokens && !a->theta) return fail(SSD_ERR_INVALID_ARG, "theta is required");
  const size_t ndt = (size_t)(p->B * p->L * p->H) * 4, nst = (size_t)(p->B * p->H * p->P * p->N) * 4;
  const size_t nx = (size_t)(p->B * p->L * p->H * p->P) * (p->io == SSD_DTYPE_BF16 ? 2 : 4);
  const Span in[] = {{a->theta, ndt, "theta"}, {a->init_state_im, nst, "init_state_im"}};
  const Span out[] = {{p->y, nx, "y"}, {p->final_state, nst, "final_state"},
                      {a->final_state_im, nst, "final_state_im"}};
  for (const Span& v : in)
    if (v.p && !aligned16(v.p)) return fail(SSD_ERR_INVALID_ARG, "%s is not 16-byte aligned", v.name);
  if (a->final_state_im && !aligned16(a->final_state_im))
    return fail(SSD_ERR_INVALID_ARG, "final_state_im is not 16-byte aligned");
  const Span base_in[] = {{p->x, nx, "x"}, {p->dt, ndt, "dt"}, {p->init, nst, "init_state"}};
  for (const Span& o : out) {
    for (const Span& v : in)
      if (overlaps(o, v)) return fail(SSD_ERR_INVALID_ARG, "%s overlaps input %s", o.name, v.name);
  }
  for (const Span& v : base_in)
    if (overlaps(out[2], v)) return fail(SSD_ERR_INVALID_ARG, "final_state_im overlaps input %s", v.name);
  if (overlaps(out[2], out[0]) || overlaps(out[2], out[1]))
    return fail(SSD_ERR_INVALID_ARG, "final_state_im overlaps another output");
  return SSD_OK;
}

}  // namespace
}  // namespace ssd

SSD_API size_t ssd_fwd_rot_workspace_size(const ssd_fwd_rot_args* a) {
  Problem p;
  if (!a || check_shape(&a->base, a->base.chunk_size, &p) != SSD_OK) return (size_t)-1;
  if (p.B == 0 || p.L == 0) return 0;
  p.complex_decay = true;
  if (rot_fused(a, p)) return fused_workspace_bytes(p);
  if (a->base.algo == SSD_ALGO_FUSED)
    return (size_t)-1;  // (the fused kernel does not take this problem)
  rot_default_chunk(a, &p);
  return rot_ws(p).total;
}

SSD_API ssd_status ssd_fwd_rot(const ssd_fwd_rot_args* a, void* stream) {
  Problem p;
  ssd_status st = rot_prologue(a, &p);
  if (st != SSD_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p.B == 0 || p.L == 0) {
    // no tokens: the final state is the initial one, real and imaginary parts
    const size_t n = (size_t)(p.B * p.H * p.P * p.N) * 4;
    cudaError_t e = cudaSuccess;
    if (p.B > 0 && p.final_state)
      e = p.init ? (p.init == p.final_state ? cudaSuccess
                                            : cudaMemcpyAsync(p.final_state, p.init, n, cudaMemcpyDeviceToDevice, s))
                 : cudaMemsetAsync(p.final_state, 0, n, s);
    if (e == cudaSuccess && p.B > 0 && p.final_im)
      e = p.init_im ? cudaMemcpyAsync(p.final_im, p.init_im, n, cudaMemcpyDeviceToDevice, s)
                    : cudaMemsetAsync(p.final_im, 0, n, s);
    return finish_launch(e, "empty-sequence state copy");
  }
  if (rot_fused(a, p)) {
    const size_t need = fused_workspace_bytes(p);
    if (!a->base.workspace || a->base.workspace_bytes < need)
      return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                  a->base.workspace ? a->base.workspace_bytes : (size_t)0);
    if (reinterpret_cast<uintptr_t>(a->base.workspace) & 255u)
      return fail(SSD_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    const size_t nst = (size_t)(p.B * p.H * p.P * p.N) * 4;
    const Span ws{a->base.workspace, need, "workspace"};
    const Span others[] = {{p.x, (size_t)(p.B * p.L * p.H * p.P) * 2, "x"},
                           {p.y, (size_t)(p.B * p.L * p.H * p.P) * 2, "y"},
                           {p.final_state, nst, "final_state"},
                           {p.final_im, nst, "final_state_im"},
                           {p.init, nst, "init_state"},
                           {p.init_im, nst, "init_state_im"},
                           {p.theta, (size_t)(p.B * p.L * p.H) * 4, "theta"}};
    for (const Span& o : others)
      if (overlaps(ws, o)) return fail(SSD_ERR_INVALID_ARG, "workspace overlaps %s", o.name);
    return finish_launch(launch_fused(p, a->base.workspace, s), "fused kernel (complex decay)");
  }
  if (a->base.algo == SSD_ALGO_FUSED)
    return fail(SSD_ERR_UNSUPPORTED, "the fused complex-decay kernel needs bf16 io, headdim 64, dstate 128, chunk 0 or 128");
  const RotWs w = rot_ws(p);
  if (!a->base.workspace || a->base.workspace_bytes < w.total)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", w.total,
                a->base.workspace ? a->base.workspace_bytes : (size_t)0);
  if (!aligned16(a->base.workspace)) return fail(SSD_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  char* ws = static_cast<char*>(a->base.workspace);
  p.err = reinterpret_cast<int32_t*>(ws);  // status word, cleared on every call
  if (cudaError_t e0 = cudaMemsetAsync(p.err, 0, sizeof(int32_t), s); e0 != cudaSuccess)
    return cuda_fail(e0, "status word");
  return finish_launch(launch_rot(p, reinterpret_cast<float*>(ws + w.off_cs), reinterpret_cast<float*>(ws + w.off_dt),
                                  reinterpret_cast<float*>(ws + w.off_phi), reinterpret_cast<float*>(ws + w.off_re),
                                  reinterpret_cast<float*>(ws + w.off_im), s,
                                  w.nbf ? ws + w.off_bf : nullptr, w.nbf ? ws + w.off_bf + w.nbf : nullptr),
                       "complex-decay forward pass");
}
