// Device status words, one per (device, caller stream).
//
// A kernel of a forward call that gives up a bounded wait, or that finds the
// cu_seqlens values inconsistent, records a code in the status word of the
// stream the call was enqueued on (every kernel of a call runs on that
// stream).  So two calls in flight on different streams cannot read,
// overwrite or clear each other's codes.  The words live in a fixed table
// compiled into the library; a stream gets a slot on its first call and keeps
// it.  Slot 0 is shared by the streams that arrive after the table is full
// (more than kStatusSlots - 1 distinct stream handles on one device).
#include <mutex>
#include <unordered_map>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

constexpr int kStatusSlots = 1024;
__device__ int g_kda_status[kStatusSlots];

namespace {

constexpr int kMaxDevices = 64;

struct StatusTable {
  std::mutex mu;
  int* base = nullptr;  // device address of g_kda_status on this device
  int next = 1;
  std::unordered_map<uintptr_t, int> slot;
};
StatusTable g_tables[kMaxDevices];

// The legacy default stream has two handles (0 and cudaStreamLegacy).
uintptr_t stream_key(cudaStream_t s) {
  return s == cudaStreamLegacy ? (uintptr_t)0 : reinterpret_cast<uintptr_t>(s);
}

}  // namespace

int* status_slot(cudaStream_t s) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  StatusTable& t = g_tables[dev];
  std::lock_guard<std::mutex> lock(t.mu);
  if (!t.base) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_kda_status) != cudaSuccess) return nullptr;
    t.base = static_cast<int*>(a);
  }
  const uintptr_t key = stream_key(s);
  auto it = t.slot.find(key);
  if (it != t.slot.end()) return t.base + it->second;
  const int idx = t.next < kStatusSlots ? t.next++ : 0;
  t.slot.emplace(key, idx);
  return t.base + idx;
}

// One block waits on an mbarrier phase that nothing completes, with the same
// bounded wait the forward kernels use, and on giving up records
// KDA_ERR_DEVICE_TIMEOUT in the status word it was given, then returns.
__global__ void kda_wait_selftest_kernel(long long limit, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(smem_u32(&bar), 0u, limit))
    atomicExch(status, KDA_ERR_DEVICE_TIMEOUT);
}

}  // namespace kda

using namespace kda;

extern "C" int kda_selftest_wait_timeout(long long cycles, void* stream) {
  if (cycles <= 0 || cycles > (1LL << 31)) return KDA_ERR_SHAPE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int* st = status_slot(s);
  if (!st) return KDA_ERR_LAUNCH;
  kda_wait_selftest_kernel<<<1, 32, 0, s>>>(cycles, st);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

extern "C" int kda_get_status(void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return -1;
  }
  int* slot = status_slot(s);
  if (!slot) return -1;
  int v = 0;
  // read, then clear, in stream order: the word reflects every call enqueued
  // on the stream before this point
  if (cudaMemcpyAsync(&v, slot, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(slot, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  return v;
}
