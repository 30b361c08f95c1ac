// Host side of libkda: argument validation, workspace layout, launches.
// Declared in include/kda.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <memory>
#include <mutex>
#include <unordered_map>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

// Exclusive prefix of per-sequence chunk counts ceil(L_n / 64), one block.
// First pass: check 0 = cu[0] <= cu[1] <= ... <= cu[N] = T.  Any violation
// sets the status word and gives every sequence zero chunks: with bounds that
// decrease somewhere, sequences can overlap and need more chunk slots than the
// workspace holds, so the chunked path then touches no token row and no slot
// (final states are still written, equal to the initial states).
__global__ void __launch_bounds__(1024) kda_chunk_offsets_kernel(const int64_t* cu, int64_t N,
                                                                  int64_t T, int64_t* chunk_off,
                                                                  int* status) {
  __shared__ int64_t warp_sums[32];
  __shared__ int64_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int bad = 0;
  for (int64_t n = tid; n <= N; n += 1024) {
    const int64_t c = cu[n];
    bad |= (n == 0 && c != 0) || (n == N && c != T) || (n > 0 && c < cu[n - 1]) || c < 0 || c > T;
  }
  const bool any_bad = __syncthreads_or(bad) != 0;
  if (tid == 0) {
    carry = 0;
    chunk_off[0] = 0;
    if (any_bad && status) atomicExch(status, 14);
  }
  __syncthreads();
  for (int64_t base = 0; base < N; base += 1024) {
    const int64_t n = base + tid;
    int64_t cnt = 0;
    if (n < N && !any_bad) cnt = (cu[n + 1] - cu[n] + kChunk - 1) / kChunk;
    int64_t x = cnt;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int64_t w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t incl = x + (warp > 0 ? warp_sums[warp - 1] : 0) + carry;
    if (n < N) chunk_off[n + 1] = incl;
    __syncthreads();
    if (tid == 1023) carry = incl;
    __syncthreads();
  }
}

void launch_chunk_offsets(const int64_t* cu, int64_t N, int64_t T, int64_t* chunk_off, int* status,
                          cudaStream_t s) {
  kda_chunk_offsets_kernel<<<1, 1024, 0, s>>>(cu, N, T, chunk_off, status);
}

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_prepared[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return p == nullptr || (((uintptr_t)p) % a) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

// Validates everything that can be checked on the host.  Returns KDA_OK or an
// error code; fills the slot count (chunk capacity) on success.
int validate(const kda_fwd_args* a, int64_t* num_slots, size_t* header_bytes) {
  if (!a) return KDA_ERR_NULL_ARG;
  const bool no_tokens = a->B == 0 || a->T == 0;  // token tensors may then be NULL (empty)
  if (!no_tokens && (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out))
    return KDA_ERR_NULL_ARG;
  if (a->K != kHeadDim || a->V != kHeadDim) return KDA_ERR_HEAD_DIM;
  if (a->B < 0 || a->T < 0 || a->H < 0 || a->N < 0 || a->H > 65535) return KDA_ERR_SHAPE;
  const uint32_t gate = a->flags & (KDA_GATE_SAFE | KDA_GATE_UNSAFE | KDA_GATE_LOGSPACE);
  if (gate != KDA_GATE_SAFE && gate != KDA_GATE_UNSAFE && gate != KDA_GATE_LOGSPACE)
    return KDA_ERR_GATE_FLAGS;
  if (a->flags & ~(KDA_GATE_SAFE | KDA_GATE_UNSAFE | KDA_GATE_LOGSPACE | KDA_QK_L2NORM |
                   KDA_BETA_PROB | KDA_G_FP32))
    return KDA_ERR_GATE_FLAGS;
  if (gate == KDA_GATE_SAFE && !(a->lower_bound >= -5.0f && a->lower_bound < 0.0f))
    return KDA_ERR_LOWER_BOUND;
  if (gate == KDA_GATE_UNSAFE && !a->A_log) return KDA_ERR_A_LOG_REQUIRED;
  if ((a->initial_state || a->final_state) && a->state_dtype != KDA_DTYPE_F32 &&
      a->state_dtype != KDA_DTYPE_BF16)
    return KDA_ERR_STATE_DTYPE;
  if (a->cu_seqlens) {
    if (a->B != 1) return KDA_ERR_VARLEN_BATCH;
  } else if (a->N != a->B) {
    return KDA_ERR_SHAPE;
  }
  if (!aligned(a->q, 16) || !aligned(a->k, 16) || !aligned(a->v, 16) || !aligned(a->g, 16) ||
      !aligned(a->out, 16) || !aligned(a->beta, 2) || !aligned(a->A_log, 4) ||
      !aligned(a->dt_bias, 16) || !aligned(a->initial_state, 16) ||
      !aligned(a->final_state, 16) || !aligned(a->cu_seqlens, 8))
    return KDA_ERR_ALIGNMENT;
  if (a->cu_seqlens) {
    *num_slots = ceil_div(a->T, kChunk) + a->N;
    *header_bytes = (size_t)(((a->N + 1) * 8 + 255) / 256 * 256);
  } else {
    *num_slots = a->B * ceil_div(a->T, kChunk);
    *header_bytes = 0;
  }
  return KDA_OK;
}

}  // namespace kda

using namespace kda;

#ifndef KDA_PIPE_RANGES
#define KDA_PIPE_RANGES 6
#endif
static_assert(KDA_PIPE_RANGES >= 1 && KDA_PIPE_RANGES <= 8, "pipeline ranges");

namespace {

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// CTAs the state stage may hold while the intra-chunk stage of the next token
// range runs beside it: half the SMs, in four 32-column CTAs per head; 0: no
// overlap.  Measured on B1 T8192 H32, where they do not fit: with 64-column
// CTAs (64 SMs) 0.314 -> 0.309 ms, within run-to-run noise; with one
// 128-column CTA per head (32 SMs, 120 left to the intra-chunk stage; 16
// epilogue warps per SM) 0.305 -> 0.365 ms, its chunk period being about
// twice as long.
int pipe_state_budget(int64_t units, int sms) { return units * 4 * 2 <= sms ? sms / 2 : 0; }

// Token ranges a dense pass is cut into (every range of every sequence, whole
// chunks), so that the state stage of range r, on a high-priority stream,
// overlaps the intra-chunk stage of range r + 1 on the SMs it leaves free:
// for few sequence-heads (above) and sequences of at least 256 chunks;
// otherwise 1.  Measured, ms per call by ranges 1 / 3 / 4 / 6 / 8: B2 T32768 H8
// 0.699 / 0.651 / 0.612 / 0.580 / 0.608, the same with H4 0.563 / 0.534 /
// 0.517 / 0.513 / 0.528; with 128 chunks per sequence (T8192, H16 or H8) no
// range count beats one pass (H8: 0.155 against 0.162 at 4 ranges).
constexpr int64_t kPipeMinChunks = 256;
int pipeline_ranges(const kda_fwd_args* a, int sms) {
  if (a->cu_seqlens || sms <= 0) return 1;
  const int64_t units = a->N * a->H;
  if (units == 0 || pipe_state_budget(units, sms) == 0) return 1;
  if (ceil_div(a->T, kChunk) < kPipeMinChunks) return 1;
  return KDA_PIPE_RANGES;
}

size_t carry_bytes(const kda_fwd_args* a) { return (size_t)(a->N * a->H) * kHeadDim * kHeadDim * 4; }

// Second stream (greatest priority) and events of the pipelined pass, one set
// per caller stream: the state stages of a call run on its caller's own
// second stream, so calls from different caller streams never share one (a
// capture open on one caller stream cannot take in another caller's work, and
// unrelated callers do not queue behind each other).
struct PipeCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t state_stream = nullptr;
  cudaEvent_t start = nullptr, end = nullptr, chunked[KDA_PIPE_RANGES] = {};
};
// At most this many caller streams per device get a second stream (kept until
// the process exits); calls from further streams run in one pass.
constexpr size_t kMaxPipeStreams = 64;
struct PipeTable {
  std::mutex mu;
  std::unordered_map<uintptr_t, std::unique_ptr<PipeCtx>> ctx;
};
PipeTable g_pipes[kMaxDevices];

bool make_pipe_ctx(PipeCtx& c) {
  if (c.ready) return true;
  int lo = 0, hi = 0;
  if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) return false;
  if (cudaStreamCreateWithPriority(&c.state_stream, cudaStreamNonBlocking, hi) != cudaSuccess) return false;
  const unsigned ef = cudaEventDisableTiming;
  if (cudaEventCreateWithFlags(&c.start, ef) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&c.end, ef) != cudaSuccess) return false;
  for (auto& e : c.chunked)
    if (cudaEventCreateWithFlags(&e, ef) != cudaSuccess) return false;
  c.ready = true;
  return true;
}

// The pipelined-pass context of caller stream `s` on device `dev`, made on
// first use; nullptr once the table is full.
PipeCtx* pipe_ctx(int dev, cudaStream_t s) {
  PipeTable& t = g_pipes[dev];
  std::lock_guard<std::mutex> lock(t.mu);
  const uintptr_t key = s == cudaStreamLegacy ? (uintptr_t)0 : reinterpret_cast<uintptr_t>(s);
  auto it = t.ctx.find(key);
  if (it != t.ctx.end()) return it->second.get();
  if (t.ctx.size() >= kMaxPipeStreams) return nullptr;
  return t.ctx.emplace(key, std::make_unique<PipeCtx>()).first->second.get();
}

}  // namespace

extern "C" size_t kda_fwd_workspace_bytes(const kda_fwd_args* args) {
  int64_t slots = 0;
  size_t header = 0;
  if (validate(args, &slots, &header) != KDA_OK) return 0;
  const size_t ws = header + (size_t)slots * (size_t)args->H * (size_t)kSlotBytes;
  return ws + (pipeline_ranges(args, device_sms()) > 1 ? carry_bytes(args) : 0);
}

int kda::fwd_device(const kda_fwd_args* a, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream, void* const* events, int init_bf16, int final_bf16,
                    bool allow_pipeline) {
  int64_t slots = 0;
  size_t header = 0;
  int rc = validate(a, &slots, &header);
  if (rc != KDA_OK) return rc;
  if (a->N == 0 || a->H == 0) return KDA_OK;
  int ranges = allow_pipeline ? pipeline_ranges(a, device_sms()) : 1;
  const size_t slot_bytes = (size_t)slots * (size_t)a->H * (size_t)kSlotBytes;
  const size_t need = header + slot_bytes + (ranges > 1 ? carry_bytes(a) : 0);
  if (need > 0 && (!workspace || !aligned(workspace, 256) || workspace_bytes < need))
    return KDA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_LAUNCH;
  if (g_prepared[dev].load() == 0) {
    if (prepare_chunk_kernel() != cudaSuccess || prepare_state_kernel() != cudaSuccess)
      return KDA_ERR_LAUNCH;
    g_prepared[dev].store(1);
  }
  // every kernel of this call reports into the status word of the caller's stream
  int* status = status_slot(stream);
  if (!status) return KDA_ERR_LAUNCH;
  PipeCtx* pipe = ranges > 1 ? pipe_ctx(dev, stream) : nullptr;
  if (!pipe) ranges = 1;  // (workspace sized for the pipelined pass is large enough for one pass)

  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  int64_t* chunk_off = a->cu_seqlens ? reinterpret_cast<int64_t*>(ws) : nullptr;
  unsigned char* slots_base = ws + header;
  void* carry = ws + header + slot_bytes;
  const int sb16 = a->state_dtype == KDA_DTYPE_BF16 ? 1 : 0;
  const int ib16 = init_bf16 >= 0 ? init_bf16 : sb16, fb16 = final_bf16 >= 0 ? final_bf16 : sb16;

  bool maps_ok = true;  // the chunk stage's tensor maps could be made
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), stream);
  };
  // The two stages over token range [t0, t0 + span) of every sequence (dense), or
  // over the whole call (packed); the range's chunks take their own workspace slots.
  auto launch_chunks = [&](int64_t t0, int64_t span, unsigned char* ws_r, cudaStream_t s,
                           int busy_sms) {
    const int64_t nt = ceil_div(span, kChunk);
    const int64_t nslots = a->cu_seqlens ? slots : a->B * nt;
    if (nslots == 0) return;
    const int64_t r0 = t0 * a->H * kHeadDim;  // element offset of the range's first row
    ChunkParams cp;
    cp.q = static_cast<const uint16_t*>(a->q) + r0;
    cp.k = static_cast<const uint16_t*>(a->k) + r0;
    cp.v = static_cast<const uint16_t*>(a->v) + r0;
    cp.g = static_cast<const uint16_t*>(a->g) + r0;
    cp.g32 = (a->flags & KDA_G_FP32) ? static_cast<const float*>(a->g) + r0 : nullptr;
    cp.beta = static_cast<const uint16_t*>(a->beta) + t0 * a->H;
    cp.A_log = a->A_log;
    cp.dt_bias = a->dt_bias;
    cp.lower_bound = a->lower_bound;
    cp.gate_mode = (a->flags & KDA_GATE_UNSAFE) ? kGateUnsafe
                   : (a->flags & KDA_GATE_LOGSPACE) ? kGateLogspace : kGateSafe;
    cp.beta_prob = (a->flags & KDA_BETA_PROB) ? 1 : 0;
    cp.l2norm = (a->flags & KDA_QK_L2NORM) ? 1 : 0;
    cp.cu = a->cu_seqlens;
    cp.chunk_off = chunk_off;
    cp.N = a->N;
    cp.T = span;
    cp.H = a->H;
    cp.NT = nt;
    cp.ld = a->T;
    cp.ws = ws_r;
    cp.status = status;
    if (!launch_chunk_kernel(cp, nslots, s, busy_sms)) maps_ok = false;
  };
  auto launch_state = [&](int64_t t0, int64_t span, unsigned char* ws_r, const void* init,
                          void* fin, int ib, int fb, cudaStream_t s) {
    const int64_t r0 = t0 * a->H * kHeadDim;
    StateParams sp;
    sp.out = static_cast<uint16_t*>(a->out) + (a->out ? r0 : 0);
    sp.init = init;
    sp.final_state = fin;
    sp.init_bf16 = ib;
    sp.final_bf16 = fb;
    sp.scale = a->scale;
    sp.cu = a->cu_seqlens;
    sp.chunk_off = chunk_off;
    sp.N = a->N;
    sp.T = span;
    sp.H = a->H;
    sp.NT = ceil_div(span, kChunk);
    sp.ld = a->T;
    sp.ws = ws_r;
    sp.status = status;
    launch_state_kernel(sp, s, ranges > 1 ? pipe_state_budget(a->N * a->H, device_sms()) : 0);
  };

  if (ranges == 1) {
    mark(0);
    if (a->cu_seqlens)
      launch_chunk_offsets(a->cu_seqlens, a->N, a->T, chunk_off, status, stream);
    launch_chunks(0, a->T, slots_base, stream, 0);
    mark(1);
    launch_state(0, a->T, slots_base, a->initial_state, a->final_state, ib16, fb16, stream);
    mark(2);
  } else {
    // chunk stage of range r on the caller's stream, state stage on the
    // high-priority stream after it; the fp32 state passes from range to range
    PipeCtx& c = *pipe;
    std::lock_guard<std::mutex> lock(c.mu);
    if (!make_pipe_ctx(c)) return KDA_ERR_LAUNCH;
    const int64_t span = ceil_div(ceil_div(a->T, kChunk), ranges) * kChunk;
    bool ok = true;
    auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
    mark(0);
    chk(cudaEventRecord(c.start, stream));
    chk(cudaStreamWaitEvent(c.state_stream, c.start, 0));
    unsigned char* ws_r = slots_base;
    int r = 0;
    for (int64_t t0 = 0; t0 < a->T; t0 += span, ++r) {
      const int64_t len = std::min(span, a->T - t0);
      const bool first = t0 == 0, last = t0 + len == a->T;
      // from the second range on, the previous range's state stage holds its SMs
      const int budget = pipe_state_budget(a->N * a->H, device_sms());
      const int state_ctas = (int)(a->N * a->H) * state_tiles(a->N * a->H, budget);
      launch_chunks(t0, len, ws_r, stream, first ? 0 : state_ctas);
      chk(cudaEventRecord(c.chunked[r], stream));
      chk(cudaStreamWaitEvent(c.state_stream, c.chunked[r], 0));
      launch_state(t0, len, ws_r, first ? a->initial_state : carry, last ? a->final_state : carry,
                   first ? ib16 : 0, last ? fb16 : 0, c.state_stream);
      ws_r += (size_t)(a->B * ceil_div(len, kChunk) * a->H) * kSlotBytes;
    }
    mark(1);
    chk(cudaEventRecord(c.end, c.state_stream));
    chk(cudaStreamWaitEvent(stream, c.end, 0));
    mark(2);
    if (!ok) return KDA_ERR_LAUNCH;
  }
  if (!maps_ok || cudaGetLastError() != cudaSuccess) return KDA_ERR_LAUNCH;
  return KDA_OK;
}

extern "C" int kda_fwd(const kda_fwd_args* a, void* workspace, size_t workspace_bytes,
                       void* stream) {
  return fwd_device(a, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr,
                    -1, -1, true);
}

extern "C" int kda_fwd_profiled(const kda_fwd_args* a, void* workspace, size_t workspace_bytes,
                                void* stream, void* const events[3]) {
  return fwd_device(a, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), events,
                    -1, -1, true);
}

extern "C" int kda_fwd_recurrent(const kda_fwd_args* a, void* stream_ptr) {
  int64_t slots = 0;
  size_t header = 0;
  const int rc = validate(a, &slots, &header);
  if (rc != KDA_OK) return rc;
  if (a->N == 0 || a->H == 0) return KDA_OK;
  RecurrentParams rp;
  rp.q = static_cast<const uint16_t*>(a->q);
  rp.k = static_cast<const uint16_t*>(a->k);
  rp.v = static_cast<const uint16_t*>(a->v);
  rp.g = static_cast<const uint16_t*>(a->g);
  rp.beta = static_cast<const uint16_t*>(a->beta);
  rp.out = static_cast<uint16_t*>(a->out);
  rp.A_log = a->A_log;
  rp.dt_bias = a->dt_bias;
  rp.lower_bound = a->lower_bound;
  rp.scale = a->scale;
  rp.gate_mode = (a->flags & KDA_GATE_UNSAFE) ? kGateUnsafe
                 : (a->flags & KDA_GATE_LOGSPACE) ? kGateLogspace : kGateSafe;
  rp.beta_prob = (a->flags & KDA_BETA_PROB) ? 1 : 0;
  rp.l2norm = (a->flags & KDA_QK_L2NORM) ? 1 : 0;
  rp.g32 = (a->flags & KDA_G_FP32) ? static_cast<const float*>(a->g) : nullptr;
  rp.init = a->initial_state;
  rp.final_state = a->final_state;
  rp.state_bf16 = a->state_dtype == KDA_DTYPE_BF16 ? 1 : 0;
  rp.cu = a->cu_seqlens;
  rp.N = a->N;
  rp.T = a->T;
  rp.H = a->H;
  rp.status = a->cu_seqlens ? status_slot(reinterpret_cast<cudaStream_t>(stream_ptr)) : nullptr;
  if (a->cu_seqlens && !rp.status) return KDA_ERR_LAUNCH;
  launch_recurrent_kernel(rp, reinterpret_cast<cudaStream_t>(stream_ptr));
  if (cudaGetLastError() != cudaSuccess) return KDA_ERR_LAUNCH;
  return KDA_OK;
}

extern "C" int kda_fwd_launches(const kda_fwd_args* a) {
  int64_t slots = 0;
  size_t header = 0;
  if (validate(a, &slots, &header) != KDA_OK || a->N == 0 || a->H == 0) return 0;
  const int ranges = pipeline_ranges(a, device_sms());
  if (ranges > 1) {  // one chunk and one state launch per token range
    const int64_t span = ceil_div(ceil_div(a->T, kChunk), ranges) * kChunk;
    return (int)(2 * ceil_div(a->T, span));
  }
  return 1 + (slots > 0 ? 1 : 0) + (a->cu_seqlens ? 1 : 0);
}

extern "C" const char* kda_error_string(int code) {
  switch (code) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL_ARG: return "a required pointer is NULL";
    case KDA_ERR_HEAD_DIM: return "K and V must both be 128";
    case KDA_ERR_SHAPE: return "invalid sizes (negative, H > 65535, or N != B without cu_seqlens)";
    case KDA_ERR_GATE_FLAGS: return "flags must select exactly one gate form and no unknown bits";
    case KDA_ERR_LOWER_BOUND: return "safe gate requires -5 <= lower_bound < 0";
    case KDA_ERR_A_LOG_REQUIRED: return "unsafe gate requires A_log";
    case KDA_ERR_STATE_DTYPE: return "state_dtype must be KDA_DTYPE_F32 or KDA_DTYPE_BF16";
    case KDA_ERR_VARLEN_BATCH: return "cu_seqlens requires B == 1";
    case KDA_ERR_ALIGNMENT: return "tensor pointers must be 16-byte aligned";
    case KDA_ERR_WORKSPACE: return "workspace missing, not 256-byte aligned, or too small";
    case KDA_ERR_LAUNCH: return "CUDA launch failed";
    case KDA_ERR_DEVICE_TIMEOUT:
      return "a kernel gave up waiting for its operand copies (device status)";
    case KDA_ERR_BAD_SEQLENS:
      return "cu_seqlens is not 0 = cu[0] <= ... <= cu[N] = T; the call skipped the sequences "
             "(device status)";
    case KDA_ERR_NOALLOC_LIMIT:
      return "problem needs more scratch than kda_fwd_noalloc's built-in buffer holds";
    default: return "unknown status code";
  }
}

extern "C" int kda_version(void) { return 100; }
