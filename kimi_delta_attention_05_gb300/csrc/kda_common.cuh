// Shared device helpers for the KDA forward kernels (sm_103a).
//
// Layout conventions
//  * A "tile128" is a [rows][128] bf16 tile in shared memory with a 256-byte
//    row pitch whose 16-byte chunks are XOR-swizzled by (row & 7), so that
//    ldmatrix reads of 8 consecutive rows hit 8 different bank groups.
//  * A "tile64" is the same for [rows][64] bf16 with a 128-byte pitch.
//  * Fragments follow the m16n8k16 bf16 mma.sync register layouts:
//      A (16x16, row-major): a0a1 = (g, 2q..2q+1), a2a3 = (g+8, ..),
//                            a4a5 = (g, 2q+8..), a6a7 = (g+8, 2q+8..)
//      B (16x8, k x n):      b0b1 = (k=2q..2q+1, n=g), b2b3 = (k=2q+8.., n=g)
//      C (16x8, fp32):       c0c1 = (g, 2q..2q+1), c2c3 = (g+8, 2q..2q+1)
//    with g = lane / 4, q = lane % 4.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kHeadDim = 128;  // K == V == 128
constexpr int kChunk = 64;     // tokens per chunk
constexpr int kSub = 16;       // tokens per diagonal sub-chunk
constexpr float kLog2e = 1.4426950408889634f;

// ---- per-(chunk, head) workspace slot ----
// Intermediates written by the chunk kernel and read by the state kernel, all
// fp16 (11-bit significand: these feed the recurrent state, where bf16's 8
// bits cost more accuracy than the tolerance allows).  Every block is stored
// as the exact shared-memory image the state kernel's tensor-core operands
// use ("kmaj" images: 128-byte-swizzled, K-major, see kmaj_off), so a chunk
// arrives with flat bulk copies.
constexpr int kSlotA1 = 0;       // kmaj R=128, K=128: rows 0-63 q gamma, rows 64-127 W
constexpr int kSlotKh = 32768;   // kmaj R=64 (t), K=128 (k): k gamma_C / gamma
constexpr int kSlotP = 49152;    // kmaj R=64 (t), K=64 (s): intra read-out matrix P
constexpr int kSlotGc = 57344;   // fp32 [128]: gamma_C
constexpr int kSlotU = 57856;    // 4 x [64 t][32 v] fp16 (chunk-swizzled, see utile_off): U per value tile
constexpr int kSlotBytes = kSlotU + 4 * 64 * 32 * 2;  // 74240 (multiple of 256)
constexpr int kSlotShared = kSlotU;                   // bytes shared by all value tiles
static_assert(kSlotBytes % 256 == 0, "slot must keep 256-byte alignment");

// Byte offset of element (row, k) in a "kmaj" image of R rows and K columns
// (K a multiple of 64): 64-column halves of R rows x 128 bytes each, the 16-byte
// chunks of a row XOR-swizzled by (row % 8).  This is the K-major layout the
// tensor cores read with the 128-byte swizzle (8-row groups 1024 bytes apart);
// read as an MN-major operand it is [K][R] with 64-wide halves R*128 bytes apart.
__device__ __forceinline__ uint32_t kmaj_off(int row, int k, int R) {
  return (uint32_t)((k >> 6) * (R * 128) + row * 128 + ((((k & 63) >> 3) ^ (row & 7)) << 4) +
                    (k & 7) * 2);
}
// Byte offset of element (t, v) (v < 32) in a U tile [64 t][32 v] fp16: 64-byte
// rows, 16-byte chunks XOR-swizzled by (t / 2) % 4 (conflict-free row reads).
__device__ __forceinline__ uint32_t utile_off(int t, int v) {
  return (uint32_t)(t * 64 + ((((v >> 3) ^ ((t >> 1) & 3))) << 4) + (v & 7) * 2);
}

// ---- swizzled shared-memory addressing ----
// A 64-row tile of 128 16-bit columns is two 8 KB halves (columns 0..63, 64..127),
// each [64 rows][128 bytes] with the 16-byte chunks of a row permuted by row % 8:
// the image a tensor copy with the 128-byte swizzle writes for a 64 x 64 box
// (at a 1024-byte aligned address), and conflict-free for 8-row matrix loads.
__device__ __forceinline__ uint32_t swz128(int row, int col) {  // byte offset
  return (uint32_t)((col >> 6) * 8192 + row * 128 + (((((col >> 3) & 7) ^ (row & 7))) << 4) +
                    ((col & 7) << 1));
}
__device__ __forceinline__ uint32_t swz64(int row, int col) {
  return (uint32_t)(row * 128 + ((((col >> 3) ^ (row & 7))) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- bf16 packing ----
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}
__device__ __forceinline__ float bf16_to_f(uint16_t u) {
  return __uint_as_float(((uint32_t)u) << 16);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
  __half2 v = *reinterpret_cast<__half2*>(&u);
  return __half22float2(v);
}

// ---- hardware approximations (single MUFU instructions) ----
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- warp-level tensor-core products (the 16 x 16 blocks of T) ----
// D += A B, m16n8k16, fp16 operands (11-bit significand), fp32 accumulation.
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// A fragment (16x16) of a 64-column swizzled tile (swz64) at (row0, col0).
__device__ __forceinline__ void lda_64(uint32_t (&a)[4], uint32_t base, int row0, int col0,
                                       int lane) {
  ldsm_x4(a, base + swz64(row0 + (lane & 15), col0 + ((lane >> 4) << 3)));
}
// B fragments for two n8 tiles (n0, n0+8) x k16 at k0, from a swz64 tile stored
// [k][n] (n contiguous), via the transposing load: b[0..1] -> tile n0,
// b[2..3] -> tile n0+8.
__device__ __forceinline__ void ldb_kn_64(uint32_t (&b)[4], uint32_t base, int n0, int k0,
                                          int lane) {
  int mi = lane >> 3;
  ldsm_x4_t(b, base + swz64(k0 + ((mi & 1) << 3) + (lane & 7), n0 + ((mi >> 1) << 3)));
}

// Pairs of fp32 values in one 64-bit register for the packed f32x2 arithmetic
// of sm_100-class SMs: one instruction per pair, each lane rounded exactly as
// the scalar instruction would (round to nearest, no flush), so results are
// bit-identical to the scalar form.  Channel pairs (c, c + 1) travel together.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 f2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f2u(f32x2 v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ---- mbarrier + bulk-copy (TMA engine) primitives ----
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(addr), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete; gives up (returns
// false) after `limit` SM cycles (default 2^31, about one second) instead of
// spinning forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity,
                                                  long long limit = 1LL << 31) {
  const long long t0 = clock64();
  while (!mbar_try_wait(addr, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}
// Flat global -> shared copy by the bulk-copy engine, completing `bytes`
// transaction bytes on the mbarrier.  Addresses and size: multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

// Tensor copy of one box of a 3-D tensor map (coordinates innermost first)
// into shared memory, completing its bytes on the mbarrier.  `map` is the
// generic address of a CUtensorMap kernel parameter (__grid_constant__).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int x, int y, int z,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(mbar)
      : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

}  // namespace kda
