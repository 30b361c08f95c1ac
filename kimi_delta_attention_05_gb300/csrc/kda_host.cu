// Forward pass on host buffers (kda_fwd_host in include/kda.h): the whole
// transfer-compute-transfer sequence of one call, pipelined in pieces so that
// the host-to-device copy of piece p + 1, the kernels of piece p and the
// device-to-host copy of piece p - 1 run at the same time.  The CPU-GPU link
// (~210 GB/s one way on this part, for copy engines and SM loads alike) is
// several times slower than the kernels, so the call costs about the link time
// of its bytes instead of link time plus compute time.
//
// Pieces: dense inputs ([B, T, H, 128]) are cut along the token axis into
// ranges of whole 64-token chunks; every piece is a dense sub-problem
// [B, span, H, 128] (gathered by 2-D copies) whose recurrent state is handed to
// the next piece in fp32 (the state stage keeps it in fp32 throughout, so the
// split does not change a single bit of the result).  Packed inputs
// (cu_seqlens) are cut between sequences, each group a varlen sub-problem.
#include <algorithm>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {
namespace {

#ifndef KDA_HOST_PIECE_MIB
#define KDA_HOST_PIECE_MIB 32
#endif
constexpr int64_t kPieceInputBytes = (int64_t)KDA_HOST_PIECE_MIB << 20;  // input bytes a piece aims at
constexpr int kMaxPieces = 64;
#ifndef KDA_HOST_H2D_STREAMS
#define KDA_HOST_H2D_STREAMS 1
#endif
// Pieces alternate over this many host-to-device streams.  Measured on the
// long-context workload (B1 T8192 H32): one stream and 32 MiB pieces 1.56 ms
// per call; 16 MiB pieces 1.65 ms (a fixed cost per piece); two or three
// streams 1.58 / 1.63 ms (copies of two pieces share the link, so each
// lands later).
constexpr int kH2dStreams = KDA_HOST_H2D_STREAMS;
constexpr int64_t kRowBytes = kHeadDim * 2;       // one bf16 [128] row
constexpr int64_t kStateElems = (int64_t)kHeadDim * kHeadDim;
constexpr int kMaxDevices = 64;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

struct Piece {
  int64_t t0, t1;  // dense: token range in every sequence; varlen: packed token range
  int64_t n0, n1;  // sequences
};

struct Plan {
  bool varlen = false;
  std::vector<Piece> pieces;
  size_t q = 0, k = 0, v = 0, g = 0, beta = 0, out = 0, alog = 0, dtb = 0, cu = 0, cur = 0, init = 0,
         fin = 0, carry = 0, ws = 0, ws_bytes = 0, total = 0;
};

// Everything kda_fwd checks, plus the host-side cu_seqlens values; then the
// pieces and the layout of the device buffer.
int make_plan(const kda_fwd_args* a, Plan* pl) {
  int64_t slots = 0;
  size_t header = 0;
  int rc = validate(a, &slots, &header);
  if (rc != KDA_OK) return rc;
  const int64_t B = a->B, T = a->T, H = a->H, N = a->N;
  const int64_t* cu = a->cu_seqlens;
  pl->varlen = cu != nullptr;
  if (cu) {
    if (cu[0] != 0 || cu[N] != T) return KDA_ERR_SHAPE;
    for (int64_t n = 0; n < N; ++n)
      if (cu[n + 1] < cu[n]) return KDA_ERR_SHAPE;
  }
  if (N == 0 || H == 0) return KDA_OK;  // nothing to move or compute
  const int64_t g_row = (a->flags & KDA_G_FP32) ? 2 * kRowBytes : kRowBytes;  // bytes of one g row
  const int64_t th_bytes = H * (3 * kRowBytes + g_row + 2);  // q, k, v, g rows and beta per token
  const int64_t total_in = B * T * th_bytes;
  const int64_t target = std::max(kPieceInputBytes, cdiv(total_in, kMaxPieces));
  size_t ws_max = 0;
  if (!cu) {
    int64_t span = T;
    if (T > 0) {
      const int64_t P = std::min<int64_t>(kMaxPieces, std::max<int64_t>(1, cdiv(total_in, target)));
      span = cdiv(cdiv(T, P), kChunk) * kChunk;
    }
    if (T == 0) pl->pieces.push_back({0, 0, 0, N});
    for (int64_t t0 = 0; t0 < T; t0 += span) pl->pieces.push_back({t0, std::min(T, t0 + span), 0, N});
    ws_max = (size_t)(B * cdiv(span, kChunk) * H) * kSlotBytes;
  } else {
    int64_t n0 = 0;
    for (int64_t n = 0; n < N; ++n) {
      const bool last = n + 1 == N;
      const bool room = (int)pl->pieces.size() < kMaxPieces - 1;
      if (last || (room && (cu[n + 1] - cu[n0]) * th_bytes >= target)) {
        pl->pieces.push_back({cu[n0], cu[n + 1], n0, n + 1});
        n0 = n + 1;
      }
    }
    for (const Piece& p : pl->pieces) {
      const int64_t ng = p.n1 - p.n0;
      const size_t w = al256((size_t)(ng + 1) * 8) +
                       (size_t)((cdiv(p.t1 - p.t0, kChunk) + ng) * H) * kSlotBytes;
      ws_max = std::max(ws_max, w);
    }
  }
  const size_t rows = (size_t)(B * T);
  const size_t esz = a->state_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t state_bytes = (size_t)(N * H * kStateElems) * esz;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += al256(bytes);
    return o;
  };
  pl->q = take(rows * H * kRowBytes);
  pl->k = take(rows * H * kRowBytes);
  pl->v = take(rows * H * kRowBytes);
  pl->g = take(rows * H * g_row);
  pl->beta = take(rows * H * 2);
  pl->out = take(rows * H * kRowBytes);
  pl->alog = take(a->A_log ? H * 4 : 0);
  pl->dtb = take(a->dt_bias ? H * kHeadDim * 4 : 0);
  pl->cu = take(cu ? (size_t)(N + 1) * 8 : 0);
  pl->cur = take(cu ? (size_t)(N + pl->pieces.size()) * 8 : 0);  // each group's cu, from 0
  pl->init = take(a->initial_state ? state_bytes : 0);
  pl->fin = take(a->final_state ? state_bytes : 0);
  pl->carry = take(!cu && pl->pieces.size() > 1 ? (size_t)(N * H * kStateElems) * 4 : 0);
  pl->ws = take(ws_max);
  pl->ws_bytes = ws_max;
  pl->total = off;
  return KDA_OK;
}

// Each packed group's cu_seqlens rebased to its first token: group i's N_i + 1
// entries at out + off[i] are cu[n0[i] + j] - cu[n0[i]].
struct RebaseTable {
  int64_t n0[kMaxPieces], n1[kMaxPieces], off[kMaxPieces];
  int count;
};
__global__ void kda_rebase_cu_kernel(const int64_t* cu, int64_t* out, RebaseTable tab) {
  for (int gi = blockIdx.x; gi < tab.count; gi += gridDim.x)
    for (int64_t j = threadIdx.x; j <= tab.n1[gi] - tab.n0[gi]; j += blockDim.x)
      out[tab.off[gi] + j] = cu[tab.n0[gi] + j] - cu[tab.n0[gi]];
}

// Per-device copy streams and events, made on first use and kept until exit.
struct HostCtx {
  std::mutex mu;
  bool ready = false;
  cudaStream_t h2d[kH2dStreams] = {}, d2h = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t loaded[kMaxPieces] = {}, computed[kMaxPieces] = {};
};
HostCtx g_ctx[kMaxDevices];

bool make_ctx(HostCtx& c) {
  if (c.ready) return true;
  const unsigned ef = cudaEventDisableTiming;
  for (int i = 0; i < kH2dStreams; ++i)
    if (cudaStreamCreateWithFlags(&c.h2d[i], cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&c.start, ef) != cudaSuccess) return false;
  if (cudaEventCreateWithFlags(&c.end, ef) != cudaSuccess) return false;
  for (int i = 0; i < kMaxPieces; ++i)
    if (cudaEventCreateWithFlags(&c.loaded[i], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&c.computed[i], ef) != cudaSuccess)
      return false;
  c.ready = true;
  return true;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_fwd_host_device_bytes(const kda_fwd_args* a) {
  Plan pl;
  if (make_plan(a, &pl) != KDA_OK) return 0;
  return pl.total;
}

extern "C" int kda_fwd_host(const kda_fwd_args* a, void* device_buffer, size_t device_bytes,
                            void* stream_ptr) {
  Plan pl;
  int rc = make_plan(a, &pl);
  if (rc != KDA_OK) return rc;
  if (pl.pieces.empty()) return KDA_OK;
  if (!device_buffer || ((uintptr_t)device_buffer & 255) || device_bytes < pl.total)
    return KDA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_LAUNCH;
  HostCtx& c = g_ctx[dev];
  std::lock_guard<std::mutex> lock(c.mu);
  if (!make_ctx(c)) return KDA_ERR_LAUNCH;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream_ptr);
  unsigned char* d = static_cast<unsigned char*>(device_buffer);
  const int64_t B = a->B, T = a->T, H = a->H, N = a->N;
  const int64_t row = H * kRowBytes, brow = H * 2;  // bytes per token: q-like, beta
  // bytes per token of q, k, v, g (g fp32 with KDA_G_FP32)
  const int64_t rows_b[4] = {row, row, row, (a->flags & KDA_G_FP32) ? 2 * row : row};
  const size_t esz = a->state_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t unit_state = (size_t)(H * kStateElems) * esz;  // one sequence's state
  const unsigned char* hq[4] = {static_cast<const unsigned char*>(a->q),
                                static_cast<const unsigned char*>(a->k),
                                static_cast<const unsigned char*>(a->v),
                                static_cast<const unsigned char*>(a->g)};
  const size_t dq[4] = {pl.q, pl.k, pl.v, pl.g};
  const unsigned char* hbeta = static_cast<const unsigned char*>(a->beta);
  unsigned char* hout = static_cast<unsigned char*>(a->out);
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  auto h2d = [&](size_t doff, const void* src, size_t bytes, cudaStream_t s) {
    if (bytes) chk(cudaMemcpyAsync(d + doff, src, bytes, cudaMemcpyHostToDevice, s));
  };
  // `rows` rows of `width` bytes between pitched layouts: one 2-D copy, or one
  // copy per row where a pitch is beyond what 2-D copies take
  int max_pitch = 0;
  chk(cudaDeviceGetAttribute(&max_pitch, cudaDevAttrMaxPitch, dev));
  auto copy_rows = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                       int64_t rows, cudaMemcpyKind kind, cudaStream_t s) {
    if (width == 0 || rows == 0) return;
    if (rows == 1) {
      chk(cudaMemcpyAsync(dst, src, width, kind, s));
    } else if (dpitch <= (size_t)max_pitch && spitch <= (size_t)max_pitch) {
      chk(cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s));
    } else {
      for (int64_t r = 0; r < rows; ++r)
        chk(cudaMemcpyAsync(static_cast<unsigned char*>(dst) + r * dpitch,
                            static_cast<const unsigned char*>(src) + r * spitch, width, kind, s));
    }
  };

  chk(cudaEventRecord(c.start, st));  // nothing is touched before earlier work on the stream
  for (int i = 0; i < kH2dStreams; ++i) chk(cudaStreamWaitEvent(c.h2d[i], c.start, 0));
  chk(cudaStreamWaitEvent(c.d2h, c.start, 0));
  // the per-call inputs go first, on the stream that also carries piece 0
  if (a->A_log) h2d(pl.alog, a->A_log, (size_t)H * 4, c.h2d[0]);
  if (a->dt_bias) h2d(pl.dtb, a->dt_bias, (size_t)H * kHeadDim * 4, c.h2d[0]);
  std::vector<int64_t> cu_off(pl.pieces.size(), 0);  // packed groups: where their cu starts
  if (a->cu_seqlens) {
    h2d(pl.cu, a->cu_seqlens, (size_t)(N + 1) * 8, c.h2d[0]);
    RebaseTable tab;
    tab.count = (int)pl.pieces.size();
    int64_t off = 0;
    for (int i = 0; i < tab.count; ++i) {
      tab.n0[i] = pl.pieces[i].n0;
      tab.n1[i] = pl.pieces[i].n1;
      tab.off[i] = cu_off[i] = off;
      off += pl.pieces[i].n1 - pl.pieces[i].n0 + 1;
    }
    kda_rebase_cu_kernel<<<tab.count, 256, 0, c.h2d[0]>>>(
        reinterpret_cast<const int64_t*>(d + pl.cu), reinterpret_cast<int64_t*>(d + pl.cur), tab);
    chk(cudaGetLastError());
  }
  if (a->initial_state) h2d(pl.init, a->initial_state, (size_t)N * unit_state, c.h2d[0]);

  const int np = (int)pl.pieces.size();
  for (int p = 0; p < np && ok; ++p) {
    const Piece& pc = pl.pieces[p];
    const int64_t span = pc.t1 - pc.t0;
    cudaStream_t hs = c.h2d[p % kH2dStreams];
    kda_fwd_args sub = *a;
    sub.A_log = a->A_log ? reinterpret_cast<const float*>(d + pl.alog) : nullptr;
    sub.dt_bias = a->dt_bias ? reinterpret_cast<const float*>(d + pl.dtb) : nullptr;
    int init_bf16 = -1, final_bf16 = -1;
    if (!pl.varlen) {
      // piece block [B, span, H, 128] at row B * t0 of the device copies
      const size_t r0 = (size_t)(B * pc.t0);
      for (int i = 0; i < 4; ++i)
        copy_rows(d + dq[i] + r0 * rows_b[i], span * rows_b[i], hq[i] + pc.t0 * rows_b[i],
                  T * rows_b[i], span * rows_b[i], B, cudaMemcpyHostToDevice, hs);
      copy_rows(d + pl.beta + r0 * brow, span * brow, hbeta + pc.t0 * brow, T * brow, span * brow,
                B, cudaMemcpyHostToDevice, hs);
      sub.q = d + pl.q + r0 * row;
      sub.k = d + pl.k + r0 * row;
      sub.v = d + pl.v + r0 * row;
      sub.g = d + pl.g + r0 * rows_b[3];
      sub.beta = d + pl.beta + r0 * brow;
      sub.out = d + pl.out + r0 * row;
      sub.T = span;
      sub.cu_seqlens = nullptr;
      const bool first = p == 0, last = p == np - 1;
      sub.initial_state = first ? (a->initial_state ? d + pl.init : nullptr) : d + pl.carry;
      sub.final_state = last ? (a->final_state ? d + pl.fin : nullptr) : d + pl.carry;
      if (!first) init_bf16 = 0;  // the carried state is fp32
      if (!last) final_bf16 = 0;
    } else {
      // sequences n0 .. n1 - 1: token rows t0 .. t1 - 1 of the packed tensors
      for (int i = 0; i < 4; ++i)
        h2d(dq[i] + pc.t0 * rows_b[i], hq[i] + pc.t0 * rows_b[i], span * rows_b[i], hs);
      h2d(pl.beta + pc.t0 * brow, hbeta + pc.t0 * brow, span * brow, hs);
      // the group as a packed call of its own: tensors from its first row, cu from 0
      sub.q = d + pl.q + pc.t0 * rows_b[0];
      sub.k = d + pl.k + pc.t0 * rows_b[1];
      sub.v = d + pl.v + pc.t0 * rows_b[2];
      sub.g = d + pl.g + pc.t0 * rows_b[3];
      sub.beta = d + pl.beta + pc.t0 * brow;
      sub.out = d + pl.out + pc.t0 * row;
      sub.cu_seqlens = reinterpret_cast<const int64_t*>(d + pl.cur) + cu_off[p];
      sub.N = pc.n1 - pc.n0;
      sub.T = span;
      sub.initial_state = a->initial_state ? d + pl.init + pc.n0 * unit_state : nullptr;
      sub.final_state = a->final_state ? d + pl.fin + pc.n0 * unit_state : nullptr;
    }
    chk(cudaEventRecord(c.loaded[p], hs));
    if (!ok) break;
    chk(cudaStreamWaitEvent(st, c.loaded[p], 0));
    rc = fwd_device(&sub, d + pl.ws, pl.ws_bytes, st, nullptr, init_bf16, final_bf16, false);
    if (rc != KDA_OK) break;
    chk(cudaEventRecord(c.computed[p], st));
    chk(cudaStreamWaitEvent(c.d2h, c.computed[p], 0));
    if (!pl.varlen) {
      copy_rows(hout + pc.t0 * row, T * row, d + pl.out + (size_t)(B * pc.t0) * row, span * row,
                span * row, B, cudaMemcpyDeviceToHost, c.d2h);
      if (p == np - 1 && a->final_state)
        chk(cudaMemcpyAsync(a->final_state, d + pl.fin, (size_t)N * unit_state,
                            cudaMemcpyDeviceToHost, c.d2h));
    } else {
      if (span > 0)
        chk(cudaMemcpyAsync(hout + pc.t0 * row, d + pl.out + pc.t0 * row, span * row,
                            cudaMemcpyDeviceToHost, c.d2h));
      if (a->final_state && pc.n1 > pc.n0)
        chk(cudaMemcpyAsync(static_cast<unsigned char*>(a->final_state) + pc.n0 * unit_state,
                            d + pl.fin + pc.n0 * unit_state, (size_t)(pc.n1 - pc.n0) * unit_state,
                            cudaMemcpyDeviceToHost, c.d2h));
    }
  }
  // the caller's stream resumes once every copy back has landed
  chk(cudaEventRecord(c.end, c.d2h));
  chk(cudaStreamWaitEvent(st, c.end, 0));
  if (rc != KDA_OK) return rc;
  return ok ? KDA_OK : KDA_ERR_LAUNCH;
}
