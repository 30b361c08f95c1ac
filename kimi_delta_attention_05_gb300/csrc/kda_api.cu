// Host side of libkda: argument validation, workspace layout, launches.
// Declared in include/kda.h.
#include <algorithm>
#include <atomic>
#include <cmath>

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

// bytes of one fp32 [N * H][128][128] state buffer
size_t state_mat_bytes(const kda_fwd_args* a) { return (size_t)(a->N * a->H) * kHeadDim * kHeadDim * 4; }

// Sequence split inside one GPU (dense calls with very few sequence-heads):
// the state stage's chain over C chunks is cut into G segments.  The state
// after a segment is affine in the state before it, S_end = S_start M + R,
// with M the state the recurrence reaches from the identity with U taken as
// zero and R the state it reaches from zero.  One launch runs segment 0 as
// usual beside the R and M runs of segments 1 .. G-1 (2G - 1 runs of C / G
// chunks at once), a small kernel chains S_{g+1} = S_g M_g + R_g, and a second
// launch runs segments 1 .. G-1 from their S_g with the outputs: 2C / G chunk
// periods instead of C.  Used when all 2G - 1 runs (four 32-column CTAs per
// sequence-head each) fit on the GPU at once for some G >= 3, with at least
// 64 chunks per segment.
#ifndef KDA_SPLIT_SEGMENTS
#define KDA_SPLIT_SEGMENTS 0  // > 0: always this many segments (measurement builds)
#endif
constexpr int kSplitMaxSegments = (kMaxStateJobs + 1) / 2;  // 2G - 1 runs in one launch
constexpr int64_t kSplitMinChunks = 64;
static_assert(KDA_SPLIT_SEGMENTS <= kSplitMaxSegments, "split segments");
int split_segments(const kda_fwd_args* a, int sms) {
  if (a->cu_seqlens || sms <= 0) return 1;
  const int64_t units = a->N * a->H, nch = ceil_div(a->T, kChunk);
  if (units == 0) return 1;
  if (KDA_SPLIT_SEGMENTS > 0) return nch >= KDA_SPLIT_SEGMENTS ? KDA_SPLIT_SEGMENTS : 1;
  for (int g = kSplitMaxSegments; g >= 3; --g)
    if ((2 * g - 1) * units * 4 <= sms && nch >= g * kSplitMinChunks) return g;
  return 1;
}
// fp32 [units][128][128] buffers of a split pass: X (segment 0's final state),
// R_g and M_g for g = 1 .. G-1, S_g for g = 2 .. G-1.
size_t split_bytes(const kda_fwd_args* a, int G) { return G > 1 ? (size_t)(3 * G - 3) * state_mat_bytes(a) : 0; }

}  // namespace

extern "C" size_t kda_fwd_workspace_bytes(const kda_fwd_args* args) {
  int64_t slots = 0;
  size_t header = 0;
  if (validate(args, &slots, &header) != KDA_OK) return 0;
  const size_t ws = header + (size_t)slots * (size_t)args->H * (size_t)kSlotBytes;
  const int sms = device_sms();
  return ws + split_bytes(args, split_segments(args, sms));
}

int kda::fwd_device(const kda_fwd_args* a, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream, void* const* events, int init_bf16, int final_bf16,
                    bool allow_split) {
  int64_t slots = 0;
  size_t header = 0;
  int rc = validate(a, &slots, &header);
  if (rc != KDA_OK) return rc;
  if (a->N == 0 || a->H == 0) return KDA_OK;
  const int G = allow_split ? split_segments(a, device_sms()) : 1;
  const size_t slot_bytes = (size_t)slots * (size_t)a->H * (size_t)kSlotBytes;
  const size_t need = header + slot_bytes + split_bytes(a, G);
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

  unsigned char* ws = reinterpret_cast<unsigned char*>(workspace);
  int64_t* chunk_off = a->cu_seqlens ? reinterpret_cast<int64_t*>(ws) : nullptr;
  unsigned char* slots_base = ws + header;
  const int sb16 = a->state_dtype == KDA_DTYPE_BF16 ? 1 : 0;
  const int ib16 = init_bf16 >= 0 ? init_bf16 : sb16, fb16 = final_bf16 >= 0 ? final_bf16 : sb16;

  bool maps_ok = true;  // the chunk stage's tensor maps could be made
  auto mark = [&](int i) {
    if (events && events[i]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[i]), stream);
  };
  // The intra-chunk stage over the whole call: every chunk takes its own workspace slot.
  auto launch_chunks = [&]() {
    if (slots == 0) return;
    ChunkParams cp;
    cp.q = static_cast<const uint16_t*>(a->q);
    cp.k = static_cast<const uint16_t*>(a->k);
    cp.v = static_cast<const uint16_t*>(a->v);
    cp.g = static_cast<const uint16_t*>(a->g);
    cp.g32 = (a->flags & KDA_G_FP32) ? static_cast<const float*>(a->g) : nullptr;
    cp.beta = static_cast<const uint16_t*>(a->beta);
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
    cp.T = a->T;
    cp.H = a->H;
    cp.NT = ceil_div(a->T, kChunk);
    cp.ld = a->T;
    cp.ws = slots_base;
    cp.status = status;
    if (!launch_chunk_kernel(cp, slots, stream)) maps_ok = false;
  };
  auto launch_state = [&](const void* init, void* fin, int ib, int fb) {
    StateParams sp;
    sp.njobs = 0;
    sp.out = static_cast<uint16_t*>(a->out);
    sp.init = init;
    sp.final_state = fin;
    sp.init_bf16 = ib;
    sp.final_bf16 = fb;
    sp.scale = a->scale;
    sp.cu = a->cu_seqlens;
    sp.chunk_off = chunk_off;
    sp.N = a->N;
    sp.T = a->T;
    sp.H = a->H;
    sp.NT = ceil_div(a->T, kChunk);
    sp.ld = a->T;
    sp.ws = slots_base;
    sp.status = status;
    launch_state_kernel(sp, stream);
  };
  // The split pass (see split_segments): runs of the state stage as jobs of one launch.
  auto launch_split = [&]() {
    const int64_t units = a->N * a->H;
    const int64_t nch = ceil_div(a->T, kChunk), segc = ceil_div(nch, G);
    const size_t mat = (size_t)units * kHeadDim * kHeadDim;  // floats per buffer
    float* X = reinterpret_cast<float*>(ws + header + slot_bytes);
    float* R = X + mat;
    float* M = R + (size_t)(G - 1) * mat;
    float* S = M + (size_t)(G - 1) * mat;
    StateParams sp;
    sp.out = static_cast<uint16_t*>(a->out);
    sp.init = nullptr;
    sp.final_state = nullptr;
    sp.init_bf16 = sp.final_bf16 = 0;
    sp.scale = a->scale;
    sp.cu = nullptr;
    sp.chunk_off = nullptr;
    sp.N = a->N;
    sp.T = a->T;
    sp.H = a->H;
    sp.NT = nch;
    sp.ld = a->T;
    sp.ws = slots_base;
    sp.status = status;
    auto job = [&](int64_t seg, const void* init, int kind, int ib, void* fin, int fb, int u_zero,
                   int write_out) {
      StateJob j;
      j.c0 = seg * segc;
      j.c1 = (seg + 1) * segc;
      j.init = init;
      j.init_kind = kind;
      j.init_bf16 = ib;
      j.fin = fin;
      j.fin_bf16 = fb;
      j.u_zero = u_zero;
      j.write_out = write_out;
      return j;
    };
    sp.njobs = 2 * G - 1;  // segment 0 as usual; R and M of the others
    sp.jobs[0] = job(0, a->initial_state, a->initial_state ? 1 : 0, ib16, X, 0, 0, 1);
    for (int g = 1; g < G; ++g) {
      sp.jobs[2 * g - 1] = job(g, nullptr, 0, 0, R + (size_t)(g - 1) * mat, 0, 0, 0);
      sp.jobs[2 * g] = job(g, nullptr, 2, 0, M + (size_t)(g - 1) * mat, 0, 1, 0);
    }
    launch_state_kernel(sp, stream);
    launch_split_combine(X, R, M, S, units, G, stream);
    sp.njobs = G - 1;  // segments 1 .. G-1 from their true initial states, with the outputs
    for (int g = 1; g < G; ++g)
      sp.jobs[g - 1] = job(g, g == 1 ? X : S + (size_t)(g - 2) * mat, 1, 0,
                           g == G - 1 ? a->final_state : nullptr, fb16, 0, 1);
    launch_state_kernel(sp, stream);
  };

  mark(0);
  if (a->cu_seqlens) launch_chunk_offsets(a->cu_seqlens, a->N, a->T, chunk_off, status, stream);
  launch_chunks();
  mark(1);
  if (G > 1) launch_split();
  else launch_state(a->initial_state, a->final_state, ib16, fb16);
  mark(2);
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
  if (split_segments(a, device_sms()) > 1) return 4;  // chunk, state, combine, state
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
