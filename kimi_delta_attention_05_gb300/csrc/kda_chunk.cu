// Intra-chunk stage of the KDA forward pass: persistent CTAs, each walking
// (64-token chunk, head) items.  Dense in-chunk products run on the 5th-
// generation tensor cores (tcgen05, operands in shared memory, fp32
// accumulators in tensor memory).
//
// For its chunk an item computes everything that does not depend on the
// recurrent state and stores it in the workspace slot of (chunk, head):
//   * the gate activation and the in-chunk cumulative decay (the "gate.py"
//     stage of the fla-kda code map: gate activation + cumulative decay),
//   * optional q/k L2 normalisation: fp32 sums of the bf16 squares on the CUDA
//     cores, taken for the next item while the current item's WY product runs,
//   * A (beta-scaled strictly-lower decayed K K^T) and P (lower decayed Q K^T)
//     from 16-token sub-chunks (fla-kda SKILL.md, "Numerical invariants"; fla-kda
//     skill page on the midpoint offset): rows carry exp(Gamma_i - Gamma_m), m the
//     midpoint of the row's sub-chunk; the diagonal sub-blocks' columns
//     exp(Gamma_m - Gamma_j), the same midpoint; the columns of an earlier
//     sub-chunk c copies exp(Gamma_e - Gamma_j) exp(Gamma_m(r) - Gamma_e) 2^64, e
//     the end of c, one copy per row sub-chunk r > c.  One product: [K xr; Q xr]
//     (128 x 128) against the 64 diagonal and the 96 off-diagonal column rows,
//   * T = (I + A)^-1: 16 x 16 diagonal inverses X_r by forward substitution in
//     fp32, the off-diagonal blocks from M_rc = -X_r A_rc and T_rc =
//     sum_m M_rm T_mc (the "solve_tril" block merges of the fla-kda code map),
//   * [W | U] = T [beta K gamma | beta V], one 128 x 256 x 64 tensor-core product
//     (the "wy_fast" WY recompute),
//   * q gamma, k gamma_C / gamma and gamma_C for the state stage.
//
// Decay factors inside a sub-chunk come from running products of
// d_t = exp(a_t), so every exponent is taken once per (token, channel).  For
// the A / P operands d_t is clamped below at exp(-10), so that the
// midpoint-relative values stay within [e^-80, e^80] for any gate; with the
// safe gate (a_t >= -5) the clamp never acts.  Where it acts, the true pair
// factor and the clamped one are both below exp(-10).  The recurrent-state
// quantities (q gamma, K gamma, k gamma_C / gamma, gamma_C) use the exact d_t.
//
// Precision: the A / P operands are bf16 (they need its exponent range), the
// diagonal inverses fp32, T and everything that feeds the recurrent state fp16
// (11-bit significand) with fp32 accumulation.
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's entry-point query)

#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "kda_kernels.cuh"
#include "kda_tc.cuh"

namespace kda {

// Tensor maps of the bf16 inputs [rows, H, 128]: 64 x 64 boxes (64 rows of one
// head, 64 channels) with the 128-byte swizzle, rows past the view zero-filled.
struct ChunkMaps {
  CUtensorMap q, k, v, g;
};

// exp(-10): floor of the per-token decay inside the A / P operands.
constexpr float kDiagDecayFloor = 4.5399929762484854e-05f;
// 2^64 and 2^-64: exact scale of the off-diagonal column copies (see the
// backward pass) and its inverse, applied to the products that use them.
constexpr float kOffScale = 18446744073709551616.0f;
constexpr float kOffScaleInv = 5.42101086242752217e-20f;

// ---- shared-memory map (bytes) ----
// Tiles of 16-bit values with 128-byte rows whose 16-byte chunks are permuted
// by row % 8: the image a tensor copy with the 128-byte swizzle writes, and the
// canonical 128-byte-swizzled operand layout of the tensor cores.
//
// Row operands, "kmaj" image of 128 rows x 128 channels (two 16 KB halves of
// 64 channels): rows 0-63 the chunk's k (raw, then bf16 k_hat xr), rows 64-127
// its q (raw, then bf16 q_hat xr).  Addressed by kmaj_off(row, ch, 128).
constexpr int kRo = 0;
// Right-hand side of the WY product, two [64 t][128 ch] tiles of two 8 KB
// halves each (swz128): raw g, then fp16 beta k_hat gamma; raw v, then fp16
// beta v.  Read as one MN-major operand of 256 columns (four 64-column blocks
// 8 KB apart).
constexpr int kRhs = 32768;
constexpr int kRhsV = kRhs + 16384;
// Column operands, kmaj image of 160 rows (two halves of 160 x 128 bytes):
// rows 0-63 k_hat yr (the diagonal sub-chunks), rows 64-159 the off-diagonal
// copies (see the backward pass), 16 rows per sub-chunk pair in the order
// (1,0) (2,0) (2,1) (3,0) (3,1) (3,2).
constexpr int kKc = 65536;
constexpr int kKcHalf = 160 * 128;
// Scratch inside the column-operand region after the A / P products (the
// column operands are dead):
constexpr int kT = kKc;              // kmaj [64][64] fp16: T = (I + A)^-1; its copy follows at +8 KB
constexpr int kAd = kKc + 20480;     // fp32 [4][16][16]: diagonal sub-blocks of A
constexpr int kA16 = kKc + 24576;    // [64][64] fp16 (swz64): off-diagonal sub-blocks of A, then M_rc
// small arrays
constexpr int kSm = kKc + 2 * kKcHalf;  // 106496
// decay products of the eight 8-token half sub-chunks, fp32 [8][2][128]: the
// exact product, then the clamped one (written by the gate stage, read by the
// operand stage; no other stage touches them)
constexpr int kCsDec = kSm;
// While the A / P product of an item runs (the decay products are dead), the
// next item's per-head gate inputs and beta inputs are staged here: fp32
// dt_bias [128], beta [64], A_log; read at the next item's start, before the
// gate stage writes the decay products.
constexpr int kStg = kCsDec;
__device__ __forceinline__ int cs_exact(int seg) { return kCsDec + seg * 1024; }
__device__ __forceinline__ int cs_clamped(int seg) { return kCsDec + seg * 1024 + 512; }
constexpr int kCsBeta = kSm + 8192;     // fp32 [64]
constexpr int kCsRq = kCsBeta + 256;    // fp32 [64]: 1 / |q| (or 1)
constexpr int kCsRk = kCsBeta + 512;    // fp32 [64]: 1 / |k| (or 1)
constexpr int kCsBar = kCsBeta + 768;   // mbarriers: q/k tiles, g/v tiles, tensor-core commits
constexpr int kCsTmem = kCsBar + 24;    // tensor-memory base address
constexpr int kChunkSmem = kCsTmem + 8;
static_assert(kRo % 1024 == 0 && kRhs % 1024 == 0 && kKc % 1024 == 0 && (kKc + kKcHalf) % 1024 == 0,
              "swizzled operand images need 1024-byte alignment");
static_assert(kChunkSmem <= 115712, "two CTAs per SM need at most 113 KB each");
constexpr uint32_t kTmemCols = 256;  // two CTAs per SM share the 512 columns

// Byte offset of (row, ch) in the column-operand image (160 rows).
__device__ __forceinline__ uint32_t kc_off(int row, int ch) {
  return (uint32_t)((ch >> 6) * kKcHalf + row * 128 + ((((ch & 63) >> 3) ^ (row & 7)) << 4) +
                    (ch & 7) * 2);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packed bf16x2 multiply (fp32 exponent range, so a factor that underflows
// does so only where the scaled value is below ~1e-38 anyway).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// The two bf16 values of a 32-bit word (low half first) as fp32.
__device__ __forceinline__ f32x2 bf2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint32_t pack_bf16_2(f32x2 v) {
  const float2 x = f2u(v);
  return pack_bf16(x.x, x.y);
}
__device__ __forceinline__ uint32_t pack_f16_2(f32x2 v) {
  const float2 x = f2u(v);
  return pack_f16(x.x, x.y);
}
__device__ __forceinline__ f32x2 max2_floor(f32x2 v) {
  const float2 x = f2u(v);
  return f2(fmaxf(x.x, kDiagDecayFloor), fmaxf(x.y, kDiagDecayFloor));
}
__device__ __forceinline__ uint32_t& u32_at(unsigned char* base, uint32_t off) {
  return *reinterpret_cast<uint32_t*>(base + off);
}

// exp(a) for the gate activation a of the pre-activation z (g + dt_bias):
//   unsafe: a = -amul softplus(z) = -amul ln(1 + e^z), so exp(a) = 2^(-amul lg2(1 + 2^(z lg2 e)));
//           for large z, 1 + 2^(.) rounds to 2^(.) and lg2 gives z lg2 e back; past the fp32
//           range it is +inf and exp(a) = 0, the limit;
//   safe:   a = lb sigmoid(amul z);
//   log-space: z is g itself, already the log decay a.
// Only exp(a) is used, so what matters is the absolute error of a: lg2(1 + t)
// loses at most ~1e-7 of it when t is tiny, far below what exp(a) resolves.
// (amul_log2e = amul lg2 e for the safe gate, amul for the unsafe one.)
// (Evaluated on a channel pair, lane by lane.)
template <int kGate>
__device__ __forceinline__ f32x2 gate_decay2(f32x2 z, float amul_log2e, float lb_log2e) {
  if (kGate == kGateLogspace) {
    const float2 a = f2u(mul2(z, f2(kLog2e, kLog2e)));
    return f2(ex2(a.x), ex2(a.y));
  }
  if (kGate == kGateUnsafe) {
    const float2 a = f2u(mul2(z, f2(kLog2e, kLog2e)));
    const float2 b = f2u(add2(f2(1.0f, 1.0f), f2(ex2(a.x), ex2(a.y))));
    const float2 c = f2u(mul2(f2(-amul_log2e, -amul_log2e), f2(lg2(b.x), lg2(b.y))));
    return f2(ex2(c.x), ex2(c.y));
  }
  const float2 a = f2u(mul2(f2(-amul_log2e, -amul_log2e), z));
  const float2 b = f2u(add2(f2(1.0f, 1.0f), f2(ex2(a.x), ex2(a.y))));
  const float2 c = f2u(mul2(f2(lb_log2e, lb_log2e), f2(rcp_approx(b.x), rcp_approx(b.y))));
  return f2(ex2(c.x), ex2(c.y));
}

// 16 x 16 product accumulated into c: A fragment a times B = block (k0.., n0..)
// of a [k][n] fp16 tile (swz64 layout).
__device__ __forceinline__ void mma16_kn(float (&c)[2][4], const uint32_t (&a)[4], uint32_t bbase,
                                         int n0, int k0, int lane) {
  uint32_t b[4];
  ldb_kn_64(b, bbase, n0, k0, lane);
  mma_f16(c[0], a, b[0], b[1]);
  mma_f16(c[1], a, b[2], b[3]);
}
// Store a 16 x 16 block held in C fragments into T (and its copy) at (r0, c0), fp16.
__device__ __forceinline__ void store_tblock(unsigned char* smem, const float (&c)[2][4], int r0,
                                             int c0, int lane) {
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t off = swz64(r0 + g + 8 * hh, c0 + 8 * nt + 2 * q4);
      const uint32_t v = pack_f16(c[nt][2 * hh], c[nt][2 * hh + 1]);
      u32_at(smem + kT, off) = v;
      u32_at(smem + kT + 8192, off) = v;
    }
}

// Store -C (a 16 x 16 block in C fragments) as fp16 at (r0, c0) of the kA16 tile.
__device__ __forceinline__ void store_mblock(unsigned char* smem, const float (&c)[2][4], int r0,
                                             int c0, int lane) {
  const int g = lane >> 2, q4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      u32_at(smem + kA16, swz64(r0 + g + 8 * hh, c0 + 8 * nt + 2 * q4)) =
          pack_f16(-c[nt][2 * hh], -c[nt][2 * hh + 1]);
}

template <int kGate, bool kL2>
__global__ void __launch_bounds__(256, 2)
    kda_chunk_kernel(ChunkParams p, int64_t num_items, const __grid_constant__ ChunkMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t H = p.H;
  const uint32_t sbase = smem_u32(smem);
  if (p.cu) num_items = p.chunk_off[p.N] * H;  // varlen: only the slots in use
  struct Item {
    int64_t slot, t0;
    int h, L;
  };
  // ---- locate a chunk: sequence n, chunk i, first token t0, length L ----
  // (32-bit divisions whenever the item count allows)
  const bool idx32 = num_items <= 0xffffffffLL;
  auto locate = [&](int64_t item) {
    Item r;
    r.slot = idx32 ? (int64_t)((uint32_t)item / (uint32_t)H) : item / H;
    r.h = (int)(item - r.slot * H);
    int64_t n, i, bos, seqlen;
    if (p.cu) {
      int64_t lo = 0, hi = p.N - 1;  // largest n with chunk_off[n] <= slot
      while (lo < hi) {
        int64_t mid = (lo + hi + 1) >> 1;
        if (p.chunk_off[mid] <= r.slot) lo = mid; else hi = mid - 1;
      }
      n = lo;
      i = r.slot - p.chunk_off[n];
      bos = p.cu[n];
      seqlen = p.cu[n + 1] - bos;
    } else {
      n = idx32 ? (int64_t)((uint32_t)r.slot / (uint32_t)p.NT) : r.slot / p.NT;
      i = r.slot - n * p.NT;
      bos = n * p.ld;
      seqlen = p.T;
    }
    r.t0 = bos + i * kChunk;
    r.L = (int)min((int64_t)kChunk, seqlen - i * kChunk);
    return r;
  };
  const uint32_t bar_qk = sbase + kCsBar, bar_gv = sbase + kCsBar + 8, bar_mma = sbase + kCsBar + 16;
  // one thread: q and k into the row-operand image (k rows 0-63, q rows 64-127)
  auto copy_qk = [&](const Item& it) {
    fence_proxy_async_smem();  // the tiles were last written by the generic proxy
    mbar_expect_tx(bar_qk, 32768u);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tma_load_3d(sbase + kRo + hh * 16384, &maps.k, 64 * hh, it.h, (int)it.t0, bar_qk);
      tma_load_3d(sbase + kRo + hh * 16384 + 8192, &maps.q, 64 * hh, it.h, (int)it.t0, bar_qk);
    }
  };
  // one thread: g (bf16 only; fp32 g is read in the gate stage) and v into the
  // right-hand-side tiles
  auto copy_gv = [&](const Item& it) {
    fence_proxy_async_smem();
    mbar_expect_tx(bar_gv, (p.g32 ? 1u : 2u) * 16384u);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (!p.g32) tma_load_3d(sbase + kRhs + hh * 8192, &maps.g, 64 * hh, it.h, (int)it.t0, bar_gv);
      tma_load_3d(sbase + kRhsV + hh * 8192, &maps.v, 64 * hh, it.h, (int)it.t0, bar_gv);
    }
  };
  // every thread: bounded wait for a barrier phase; a wait that gives up sets
  // the status word, and the item goes on with whatever the tiles hold
  bool gave_up = false;
  auto wait_bar = [&](uint32_t bar, uint32_t parity) {
    if (!gave_up && !mbar_wait_bounded(bar, parity)) {
      gave_up = true;
      atomicExch(p.status, 13);
    }
  };
  uint32_t mma_count = 0;  // commits waited on so far (phase parity of bar_mma)
  auto wait_mma = [&]() {
    wait_bar(bar_mma, mma_count & 1u);
    ++mma_count;
    tc_fence_after();
  };
  // rows L..63 copied past a short chunk's end (the next sequence's rows, or
  // zeros past the view) are cleared: the stages below expect zeros.  Tiles
  // 0, 1: k and q; 2, 3: g and v.
  auto zero_tails = [&](int L, int tile0) {
    const int n = (kChunk - L) * 16;  // 16-byte chunks per tile
    for (int idx = tid; idx < 2 * n; idx += 256) {
      const int tile = tile0 + (idx >= n), e = idx - (idx >= n ? n : 0);
      const int t = L + (e >> 4), c = 8 * (e & 15);
      uint32_t off;
      if (tile == 0) off = kRo + kmaj_off(t, c, 128);
      else if (tile == 1) off = kRo + kmaj_off(64 + t, c, 128);
      else if (tile == 2) off = kRhs + swz128(t, c);
      else off = kRhsV + swz128(t, c);
      *reinterpret_cast<uint4*>(smem + off) = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  int64_t item = blockIdx.x;
  if (item >= num_items) return;
  Item cur = locate(item);
  float* sBeta = reinterpret_cast<float*>(smem + kCsBeta);
  float* sRq = reinterpret_cast<float*>(smem + kCsRq);
  float* sRk = reinterpret_cast<float*>(smem + kCsRk);
  float* sStg = reinterpret_cast<float*>(smem + kStg);
  // an item's per-head gate inputs and beta inputs into the staging area, by
  // threads 64.. (u = tid - 64: dt_bias u < 32, A_log u = 32, beta 64 <= u < 128)
  auto stage_scalars = [&](const Item& x) {
    const int u = tid - 64;
    if (u >= 0 && u < 32)
      *reinterpret_cast<float4*>(sStg + 4 * u) =
          (p.dt_bias && kGate != kGateLogspace)
              ? __ldg(reinterpret_cast<const float4*>(p.dt_bias + x.h * kHeadDim) + u)
              : make_float4(0.f, 0.f, 0.f, 0.f);
    else if (u == 32)
      sStg[192] = (p.A_log && kGate != kGateLogspace) ? __ldg(p.A_log + x.h) : 0.f;
    else if (u >= 64 && u < 64 + kChunk)
      sStg[128 + u - 64] = u - 64 < x.L ? bf16_to_f(p.beta[(x.t0 + u - 64) * H + x.h]) : 0.f;
  };
  // An item's q and k rows once their copy has landed (parity of its phase):
  // rows past its end cleared, then the reciprocal norms 1 / sqrt(|x|^2 + eps)
  // (1 without the L2 norm) into sRk / sRq: two threads per row, 64 channels
  // each, fp32 sums of the bf16 squares (16-byte chunks taken in swizzled
  // order, so the eight rows of a group read eight different bank groups).
  auto prep_rows = [&](const Item& x, uint32_t parity) {
    wait_bar(bar_qk, parity);
    if (x.L < kChunk) zero_tails(x.L, 0);
    if (kL2) {
      __syncthreads();  // the cleared rows are read below
      const int row = tid >> 1, hh = tid & 1;
      const unsigned char* src = smem + kRo + hh * 16384 + row * 128;
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 w = *reinterpret_cast<const uint4*>(src + 16 * (c ^ (row & 7)));
        const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = f2u(bf2_to_f2(ws4[e]));
          acc.x = fmaf(f.x, f.x, acc.x);
          acc.y = fmaf(f.y, f.y, acc.y);
        }
      }
      float ss = acc.x + acc.y;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      if (hh == 0) (row < 64 ? sRk : sRq)[row & 63] = rsqrtf(ss + 1e-6f);
    } else if (tid < 128) {
      (tid < 64 ? sRk : sRq)[tid & 63] = 1.0f;
    }
  };
  stage_scalars(cur);
  if (tid == 0) {
    mbar_init(bar_qk, 1);
    mbar_init(bar_gv, 1);
    mbar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     sbase + kCsTmem),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kCsTmem);
  if (tid == 0) {
    copy_qk(cur);
    copy_gv(cur);
  }
  prep_rows(cur, 0u);
  // exact product of half s2, clamped products of the first (Xm) and second
  // (Ym) half of sub-chunk r, channels c .. c + 3
  auto ld_exact = [&](int s2, int c) { return *reinterpret_cast<const float4*>(smem + cs_exact(s2) + c * 4); };
  auto ld_xm = [&](int r, int c) { return *reinterpret_cast<const float4*>(smem + cs_clamped(2 * r) + c * 4); };
  auto ld_ym = [&](int r, int c) { return *reinterpret_cast<const float4*>(smem + cs_clamped(2 * r + 1) + c * 4); };
  // tensor-core operand descriptors (the 14-bit address field takes the
  // k-step offsets by plain addition)
  const uint64_t dRo = smem_desc(sbase + kRo, 16, 1024);
  const uint64_t dKc = smem_desc(sbase + kKc, 16, 1024);
  const uint64_t dT = smem_desc(sbase + kT, 16, 1024);
  const uint64_t dRhs = smem_desc(sbase + kRhs, 8192, 1024);

  int it = 0;
  for (; item < num_items; item += gridDim.x, ++it) {
  const int L = cur.L;
  const int h = cur.h;
  unsigned char* ws = p.ws + (cur.slot * H + h) * (int64_t)kSlotBytes;
  const int64_t next = item + gridDim.x;
  Item nxt = cur;  // located while the A / P product runs
  // this item's staged per-head gate inputs (this thread's four channels) and beta
  const float4 dtb = *reinterpret_cast<const float4*>(sStg + 4 * (tid & 31));
  const float alog = sStg[192];
  if (tid < kChunk) {
    const float bl = sStg[128 + tid];
    sBeta[tid] = tid >= L ? 0.f : (p.beta_prob ? bl : rcp_approx(1.0f + ex2(-bl * kLog2e)));
  }
  // (this item's q, k copy was waited on, and its rows prepared, one item ahead)
  wait_bar(bar_gv, (uint32_t)(it & 1));
  if (L < kChunk) zero_tails(L, 2);
  fence_proxy_async_smem();  // the zeroed rows are read by the tensor core later
  tc_fence_before();
  __syncthreads();

  // ---- gate activation, per-token decays d (registers), half sub-chunk products ----
  // thread -> sub-chunk rb, half hf (tokens 8 hf .. 8 hf + 7 of it), channels c0 .. c0 + 3;
  // a warp covers all 128 channels of one half, so every token row is one access
  const int cg = tid & 31, hf = (tid >> 5) & 1, rb = tid >> 6;
  const int c0 = 4 * cg;
  const int seg = 2 * rb + hf;      // half sub-chunk index 0..7
  const int tb = 16 * rb + 8 * hf;  // its first token
  f32x2 d2[8][2];  // decays of channel pairs (c0, c0 + 1), (c0 + 2, c0 + 3)
  float inv[4];    // 1 / (clamped product over this half)
  const f32x2 one2 = f2(1.0f, 1.0f);
  {
    const f32x2 dtb2[2] = {f2(dtb.x, dtb.y), f2(dtb.z, dtb.w)};
    const float amul_log2e = (p.A_log && kGate != kGateLogspace ? expf(alog) : 1.0f) *
                             (kGate == kGateUnsafe ? 1.0f : kLog2e);
    const float lb_log2e = p.lower_bound * kLog2e;
    f32x2 D2[2] = {one2, one2}, Dc2[2] = {one2, one2};
    auto gate_token = [&](int j, f32x2 g01, f32x2 g23) {
      const int t = tb + j;
      const f32x2 gz[2] = {g01, g23};
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        f32x2 e = gate_decay2<kGate>(add2(gz[pp], dtb2[pp]), amul_log2e, lb_log2e);
        if (t >= L) e = one2;
        d2[j][pp] = e;
        D2[pp] = mul2(D2[pp], e);
        Dc2[pp] = mul2(Dc2[pp], max2_floor(e));
      }
    };
    if (p.g32) {  // fp32 g straight from global memory, four tokens' loads in flight at a time
#pragma unroll
      for (int j0 = 0; j0 < 8; j0 += 4) {
        float4 gv[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int t = tb + j0 + jj;
          gv[jj] = t < L ? __ldg(reinterpret_cast<const float4*>(p.g32 + ((cur.t0 + t) * H + h) * kHeadDim + c0))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          gate_token(j0 + jj, f2(gv[jj].x, gv[jj].y), f2(gv[jj].z, gv[jj].w));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint2 graw = *reinterpret_cast<const uint2*>(smem + kRhs + swz128(tb + j, c0));
        gate_token(j, bf2_to_f2(graw.x), bf2_to_f2(graw.y));
      }
    }
    const float2 Da = f2u(D2[0]), Db = f2u(D2[1]), Dca = f2u(Dc2[0]), Dcb = f2u(Dc2[1]);
    *reinterpret_cast<float4*>(smem + cs_exact(seg) + c0 * 4) = make_float4(Da.x, Da.y, Db.x, Db.y);
    *reinterpret_cast<float4*>(smem + cs_clamped(seg) + c0 * 4) = make_float4(Dca.x, Dca.y, Dcb.x, Dcb.y);
    // (an approximate reciprocal: it only scales the bf16 A / P operands)
    inv[0] = rcp_approx(Dca.x);
    inv[1] = rcp_approx(Dca.y);
    inv[2] = rcp_approx(Dcb.x);
    inv[3] = rcp_approx(Dcb.y);
  }
  __syncthreads();  // the half products are read by every warp below

  // ---- operands ----
  //  exact, chunk relative:     gamma_j = prod_{s<=j} d_s  -> beta K gamma (rhs), q gamma (ws)
  //  exact, chunk-end relative: gamma_C / gamma_j           -> k_hat (ws)
  //  clamped, midpoint relative: xr_j = e^{lam_j - lam_7}, yr_j = 1 / xr_j -> A / P operands;
  //  within the half before the midpoint xr_j = inv * (clamped product up to j), after
  //  it xr_j = clamped product from token 8 up to j, so each half needs only its own d
  f32x2 pre2[2] = {one2, one2}, suf2[2] = {one2, one2};
#pragma unroll
  for (int s2 = 0; s2 < 8; ++s2) {
    const float4 Ds = ld_exact(s2, c0);
    const f32x2 dv2[2] = {f2(Ds.x, Ds.y), f2(Ds.z, Ds.w)};
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      if (s2 < seg) pre2[pp] = mul2(pre2[pp], dv2[pp]);
      if (s2 > seg) suf2[pp] = mul2(suf2[pp], dv2[pp]);
    }
  }
  if (tid < 32) {
    // gamma_C = product over all eight halves
    const float2 sa = f2u(suf2[0]), sbv = f2u(suf2[1]);
    const float4 D0 = ld_exact(0, c0);
    *reinterpret_cast<float4*>(ws + kSlotGc + c0 * 4) =
        make_float4(sa.x * D0.x, sa.y * D0.y, sbv.x * D0.z, sbv.y * D0.w);
  }
  // xr takes 1 / (clamped product) in the first half, yr in the second
  const f32x2 invx2[2] = {hf ? one2 : f2(inv[0], inv[1]), hf ? one2 : f2(inv[2], inv[3])};
  const f32x2 inv2[2] = {hf ? f2(inv[0], inv[1]) : one2, hf ? f2(inv[2], inv[3]) : one2};
  // backward over the half (reads the raw k): k_hat (ws), the diagonal column
  // operand and the off-diagonal column copies.  The copy of row j (sub-chunk rb)
  // for row sub-chunk r > rb is k_hat_j sigma_j Phi_r with sigma_j = e^{lam_e - lam_j}
  // relative to the end e of sub-chunk rb and Phi_r = 2^64 e^{lam_m(r) - lam_e} (the
  // first half of r and the sub-chunks in between): every factor is <= 1 apart from
  // the exact 2^64, so a factor that underflows does so only where the entry it
  // builds is negligible, while the midpoint-relative row operand (up to e^70)
  // still finds its partner; the epilogue takes the 2^64 back out.
  {
    unsigned char* gKh = ws + kSlotKh;
    f32x2 phi[3][2];
    {
      float4 ph[3];
#pragma unroll
      for (int r = 1; r < 4; ++r) {
        if (r > rb) {
          float4 e = ld_xm(r, c0);
          e.x *= kOffScale;
          e.y *= kOffScale;
          e.z *= kOffScale;
          e.w *= kOffScale;
#pragma unroll
          for (int s3 = 1; s3 < 3; ++s3) {
            if (s3 > rb && s3 < r) {
              const float4 xm = ld_xm(s3, c0);
              const float4 ym = ld_ym(s3, c0);
              e.x *= xm.x * ym.x;
              e.y *= xm.y * ym.y;
              e.z *= xm.z * ym.z;
              e.w *= xm.w * ym.w;
            }
          }
          ph[r - 1] = e;
        } else {
          ph[r - 1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        phi[r - 1][0] = f2(ph[r - 1].x, ph[r - 1].y);
        phi[r - 1][1] = f2(ph[r - 1].z, ph[r - 1].w);
      }
    }
    // sigma_j = (clamped product from j + 1 to the end of the half) x (second-half
    // product of the sub-chunk, in the first half)
    f32x2 sig2[2] = {one2, one2};
    if (!hf) {
      const float4 ym = ld_ym(rb, c0);
      sig2[0] = f2(ym.x, ym.y);
      sig2[1] = f2(ym.z, ym.w);
    }
    f32x2 y2[2] = {suf2[0], suf2[1]}, yc2[2] = {one2, one2};
#pragma unroll
    for (int j = 7; j >= 0; --j) {
      const int t = tb + j;
      const float rk = sRk[t];
      const f32x2 rk2 = f2(rk, rk);
      const uint2 kraw = *reinterpret_cast<const uint2*>(smem + kRo + kmaj_off(t, c0, 128));
      const f32x2 k2[2] = {mul2(bf2_to_f2(kraw.x), rk2), mul2(bf2_to_f2(kraw.y), rk2)};
      const f32x2 yr2[2] = {mul2(yc2[0], inv2[0]), mul2(yc2[1], inv2[1])};  // inv = 1 in the first half
      *reinterpret_cast<uint2*>(smem + kKc + kc_off(t, c0)) =
          make_uint2(pack_bf16_2(mul2(k2[0], yr2[0])), pack_bf16_2(mul2(k2[1], yr2[1])));
      *reinterpret_cast<uint2*>(gKh + kmaj_off(t, c0, 64)) =
          make_uint2(pack_f16_2(mul2(k2[0], y2[0])), pack_f16_2(mul2(k2[1], y2[1])));
      const f32x2 ks2[2] = {mul2(k2[0], mul2(yc2[0], sig2[0])), mul2(k2[1], mul2(yc2[1], sig2[1]))};
#pragma unroll
      for (int r = 1; r < 4; ++r) {
        if (r > rb) {
          const int row = 64 + 16 * (r * (r - 1) / 2 + rb) + (t & 15);  // pair (r, rb)
          *reinterpret_cast<uint2*>(smem + kKc + kc_off(row, c0)) =
              make_uint2(pack_bf16_2(mul2(ks2[0], phi[r - 1][0])), pack_bf16_2(mul2(ks2[1], phi[r - 1][1])));
        }
      }
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        y2[pp] = mul2(y2[pp], d2[j][pp]);
        yc2[pp] = mul2(yc2[pp], max2_floor(d2[j][pp]));
      }
    }
  }
  // forward over the half (overwrites raw q, k, g, v).  No barrier: from the
  // gate stage on, every thread reads and writes only its own elements of the
  // q, k, g and v tiles.

  {
    unsigned char* gQg = ws + kSlotA1;  // rows 0..63 of the [q gamma; W] image
    f32x2 x2[2] = {pre2[0], pre2[1]}, xc2[2] = {one2, one2};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = tb + j;
      const uint32_t ok = kRo + kmaj_off(t, c0, 128), oq = ok + 8192;  // rows t and 64 + t
      const uint32_t og = swz128(t, c0);
      f32x2 xr2[2];
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        x2[pp] = mul2(x2[pp], d2[j][pp]);
        xc2[pp] = mul2(xc2[pp], max2_floor(d2[j][pp]));
        xr2[pp] = mul2(xc2[pp], invx2[pp]);  // invx = 1 in the second half
      }
      const float rk = sRk[t], rq = sRq[t], bt = sBeta[t];
      const f32x2 rk2 = f2(rk, rk), rq2 = f2(rq, rq), bt2 = f2(bt, bt);
      const uint2 kraw = *reinterpret_cast<const uint2*>(smem + ok);
      const uint2 qraw = *reinterpret_cast<const uint2*>(smem + oq);
      const uint2 vraw = *reinterpret_cast<const uint2*>(smem + kRhsV + og);
      const f32x2 k2[2] = {mul2(bf2_to_f2(kraw.x), rk2), mul2(bf2_to_f2(kraw.y), rk2)};
      const f32x2 q2[2] = {mul2(bf2_to_f2(qraw.x), rq2), mul2(bf2_to_f2(qraw.y), rq2)};
      const f32x2 v2[2] = {bf2_to_f2(vraw.x), bf2_to_f2(vraw.y)};
      *reinterpret_cast<uint2*>(smem + ok) =
          make_uint2(pack_bf16_2(mul2(k2[0], xr2[0])), pack_bf16_2(mul2(k2[1], xr2[1])));
      *reinterpret_cast<uint2*>(smem + oq) =
          make_uint2(pack_bf16_2(mul2(q2[0], xr2[0])), pack_bf16_2(mul2(q2[1], xr2[1])));
      *reinterpret_cast<uint2*>(smem + kRhs + og) =
          make_uint2(pack_f16_2(mul2(mul2(bt2, k2[0]), x2[0])), pack_f16_2(mul2(mul2(bt2, k2[1]), x2[1])));
      *reinterpret_cast<uint2*>(smem + kRhsV + og) =
          make_uint2(pack_f16_2(mul2(bt2, v2[0])), pack_f16_2(mul2(bt2, v2[1])));
      *reinterpret_cast<uint2*>(gQg + kmaj_off(t, c0, 128)) =
          make_uint2(pack_f16_2(mul2(q2[0], x2[0])), pack_f16_2(mul2(q2[1], x2[1])));
    }
  }
  fence_proxy_async_smem();  // the operands are read by the tensor core next
  tc_fence_before();
  __syncthreads();

  // ---- A / P product: [K xr; Q xr] (128 x 128) against all 160 column-operand rows:
  //      tensor-memory columns 0..63 the diagonal, 64..159 the off-diagonal copies ----
  if (warp == 0) {
    tc_fence_after();
    const uint32_t id = idesc_bf16(128, 160, false, false);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint64_t oa = (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4);
      const uint64_t ob = (uint64_t)(((ks >> 2) * kKcHalf + (ks & 3) * 32) >> 4);
      tc_mma(tmem, dRo + oa, dKc + ob, id, ks > 0);
    }
    tc_commit(bar_mma);
  }
  if (next < num_items) nxt = locate(next);  // while the tensor core runs
  wait_mma();
  // q, k tiles are free: the next item's q, k
  if (next < num_items && tid == 0) copy_qk(nxt);
  // ---- A / P epilogue: lane = row of [K xr; Q xr]; rows 0..63 give A (beta-scaled,
  //      strictly lower), rows 64..127 P (lower).  Warps w and w + 4 share a lane
  //      quarter: w < 4 the diagonal sub-block (and, for sub-chunks 2 and 3, the
  //      first two off-diagonal pieces), w >= 4 the other off-diagonal pieces ----
  {
    const int qd = warp & 3, hw = warp >> 2;
    const int row = 32 * qd + lane;
    const bool isA = row < 64;
    const int i = row & 63, r = i >> 4, ii = i & 15;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
    unsigned char* gP = ws + kSlotP;  // kmaj image R=64, K=64
    const float bt = isA ? sBeta[i] : 1.f;
    if (hw == 0) {
      float v[32];
      tc_ld32(lane_base + 32 * (qd & 1), v);
      float e[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float x = (r & 1) ? v[16 + j] : v[j];
        e[j] = isA ? (j < ii ? x * bt : 0.f) : (j <= ii ? x : 0.f);
      }
      if (isA) {
        float4* ad = reinterpret_cast<float4*>(smem + kAd + (r * 256 + ii * 16) * 4);
#pragma unroll
        for (int c = 0; c < 4; ++c) ad[c] = make_float4(e[4 * c], e[4 * c + 1], e[4 * c + 2], e[4 * c + 3]);
      } else {
        // P columns 16 r .. 16 r + 15 (the zeros right of them are written above)
#pragma unroll
        for (int c = 0; c < 2; ++c)
          *reinterpret_cast<uint4*>(gP + kmaj_off(i, 16 * r + 8 * c, 64)) =
              make_uint4(pack_f16(e[8 * c], e[8 * c + 1]), pack_f16(e[8 * c + 2], e[8 * c + 3]),
                         pack_f16(e[8 * c + 4], e[8 * c + 5]), pack_f16(e[8 * c + 6], e[8 * c + 7]));
      }
    }
    // off-diagonal columns 0 .. 16 r - 1 of row i sit at tensor-memory columns
    // 64 + 8 r (r - 1) + j; taken in 16-column pieces (column, sub-chunk, first j):
    // quarters of sub-chunks 0, 1: (64, 1, 0); of sub-chunks 2, 3: (80, 2, 0) (96, 2, 16)
    // (112, 3, 0) (128, 3, 16) (144, 3, 32).  Sub-chunk 2's two pieces go to the warp
    // that did the diagonal part.
    const int pc0 = (qd & 1) ? (hw == 0 ? 0 : 2) : 0;
    const int pc1 = (qd & 1) ? (hw == 0 ? 2 : 5) : (hw == 0 ? 0 : 1);
    for (int pc = pc0; pc < pc1; ++pc) {
      const int col = (qd & 1) ? 80 + 16 * pc : 64;
      const int blk = (qd & 1) ? (pc < 2 ? 2 : 3) : 1;
      const int j0 = (qd & 1) ? 16 * (pc < 2 ? pc : pc - 2) : 0;
      float a[16];
      tc_ld16(lane_base + col, a);
      if (r == blk) {
        const float sc = (isA ? bt : 1.f) * kOffScaleInv;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 val = make_uint4(pack_f16(sc * a[8 * c], sc * a[8 * c + 1]), pack_f16(sc * a[8 * c + 2], sc * a[8 * c + 3]),
                                       pack_f16(sc * a[8 * c + 4], sc * a[8 * c + 5]), pack_f16(sc * a[8 * c + 6], sc * a[8 * c + 7]));
          if (isA) *reinterpret_cast<uint4*>(smem + kA16 + swz64(i, j0 + 8 * c)) = val;
          else *reinterpret_cast<uint4*>(gP + kmaj_off(i, j0 + 8 * c, 64)) = val;
        }
      }
    }
    // zero the blocks of T above the diagonal (sub-block pairs (r, c), c > r), both copies
    for (int idx = tid; idx < 2 * 6 * 16 * 2; idx += 256) {
      const int cp = idx / 192, e = idx - cp * 192;
      const int pr = e >> 5, rr = (e >> 1) & 15, hh = e & 1;  // pair, row, 8-column half
      const int br = pr < 3 ? 0 : (pr < 5 ? 1 : 2);
      const int bc = br + 1 + (pr - (br == 0 ? 0 : (br == 1 ? 3 : 5)));
      *reinterpret_cast<uint4*>(smem + kT + cp * 8192 + swz64(16 * br + rr, 16 * bc + 8 * hh)) =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }
  tc_fence_before();
  __syncthreads();

  // ---- X_r = (I + A_rr)^-1 by forward substitution (warp w: sub-chunks 2 w and
  //      2 w + 1 in lanes 0-15 and 16-31, lane = column) into the diagonal blocks of T ----
  if (warp < 2) {
    const int j = lane & 15, rx = 2 * warp + (lane >> 4);
    const float4* Ad4 = reinterpret_cast<const float4*>(smem + kAd + rx * 1024);  // rows of 16 floats
    float x[kSub];
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: a short dependency chain
#pragma unroll
      for (int s4 = 0; 4 * s4 < ii; ++s4) {  // row ii, four entries per 16-byte load
        const float4 a = Ad4[ii * 4 + s4];
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (4 * s4 + c < ii) acc[c] += av[c] * x[4 * s4 + c];
      }
      x[ii] = (ii == j) ? 1.f : (ii < j ? 0.f : -((acc[0] + acc[1]) + (acc[2] + acc[3])));
    }
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii) {
      const __half xv = __float2half_rn(x[ii]);
      const uint32_t off = swz64(16 * rx + ii, 16 * rx + j);
      *reinterpret_cast<__half*>(smem + kT + off) = xv;
      *reinterpret_cast<__half*>(smem + kT + 8192 + off) = xv;
    }
  } else {
    // the other warps meanwhile: the next item's scalars into the staging area
    // (the decay products are dead), and the columns of P right of each row's
    // sub-chunk, which are zero
    if (next < num_items) stage_scalars(nxt);
    if (tid >= 192) {
      const int i = tid - 192, r = i >> 4;
      for (int c = 2 * r + 2; c < 8; ++c)
        *reinterpret_cast<uint4*>(ws + kSlotP + kmaj_off(i, 8 * c, 64)) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  __syncthreads();
  // ---- off-diagonal blocks of T: T_rc = sum_{m=c}^{r-1} M_rm T_mc, M_rm = -X_r A_rm.
  //      Level 0: six warps form one M_rc each (fp16, over A_rc in place).  Level 1:
  //      T_10, T_21, T_32 = M_r,r-1 X_r-1, while three warps start the sums of T_20,
  //      T_31 and T_30 (fp32 fragments in registers).  Levels 2 and 3 add the terms
  //      whose T blocks the previous level stored.  Every block keeps one accumulator
  //      fed in the order m = c .. r - 1. ----
  if (warp < 6) {
    const int r = warp < 1 ? 1 : (warp < 3 ? 2 : 3), c = warp - (r * (r - 1)) / 2;
    uint32_t xa[4];
    lda_64(xa, sbase + kT, 16 * r, 16 * r, lane);  // X_r
    float acc[2][4] = {};
    mma16_kn(acc, xa, sbase + kA16, 16 * c, 16 * r, lane);  // X_r A_rc
    store_mblock(smem, acc, 16 * r, 16 * c, lane);
  }
  __syncthreads();
  float tacc[2][4] = {};  // warp 3: T_20, warp 4: T_31, warp 5: T_30 (partial sums)
  if (warp < 6) {
    uint32_t am[4];
    if (warp < 3) {  // T_r,r-1 = M_r,r-1 X_r-1, r = warp + 1
      const int r = warp + 1;
      lda_64(am, sbase + kA16, 16 * r, 16 * (r - 1), lane);
      float t[2][4] = {};
      mma16_kn(t, am, sbase + kT, 16 * (r - 1), 16 * (r - 1), lane);
      store_tblock(smem, t, 16 * r, 16 * (r - 1), lane);
    } else {  // first terms: M_20 X_0, M_31 X_1, M_30 X_0
      const int r = warp == 4 ? 3 : (warp == 3 ? 2 : 3), c = warp == 4 ? 1 : 0;
      lda_64(am, sbase + kA16, 16 * r, 16 * c, lane);
      mma16_kn(tacc, am, sbase + kT, 16 * c, 16 * c, lane);
    }
  }
  __syncthreads();
  if (warp >= 3 && warp < 6) {  // + M_21 T_10 (T_20), M_32 T_21 (T_31), M_31 T_10 (T_30)
    const int r = warp == 3 ? 2 : 3, m = warp == 4 ? 2 : 1, c = warp == 4 ? 1 : 0;
    uint32_t am[4];
    lda_64(am, sbase + kA16, 16 * r, 16 * m, lane);
    mma16_kn(tacc, am, sbase + kT, 16 * c, 16 * m, lane);
    if (warp < 5) store_tblock(smem, tacc, 16 * r, 16 * c, lane);
  }
  __syncthreads();
  if (warp == 5) {  // T_30 += M_32 T_20
    uint32_t am[4];
    lda_64(am, sbase + kA16, 48, 32, lane);
    mma16_kn(tacc, am, sbase + kT, 0, 32, lane);
    store_tblock(smem, tacc, 48, 0, lane);
  }
  fence_proxy_async_smem();  // T is read by the tensor core next
  tc_fence_before();
  __syncthreads();

  // ---- [W | U] = T [beta K gamma | beta V]: M = 128 (rows 64.. repeat T), N = 256, K = 64 ----
  if (warp == 0) {
    tc_fence_after();
    const uint32_t id = idesc_f16(128, 256, false, true);
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      tc_mma(tmem, dT + (uint64_t)((ks * 32) >> 4), dRhs + (uint64_t)((ks * 2048) >> 4), id, ks > 0);
    tc_commit(bar_mma);
  }
  // while the tensor core runs: the next item's q, k rows and norms (its copy
  // went out after the A / P product; this item's norms are no longer read)
  if (next < num_items) prep_rows(nxt, (uint32_t)((it + 1) & 1));
  wait_mma();
  // the right-hand-side tiles are free: the next item's g and v
  if (next < num_items && tid == 0) copy_gv(nxt);
  // ---- W and U rows: lane quarter qd holds rows (32 qd + lane) % 64; quarters 0, 1
  //      write W, quarters 2, 3 write U, each warp 64 of its 128 columns ----
  {
    const int qd = warp & 3, hw = warp >> 2;
    const int i = (32 * qd + lane) & 63;
    const bool isW = qd < 2;
    const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + (isW ? 0 : 128) + 64 * hw;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
      tc_ld32(taddr + 32 * half, v);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int col = 64 * hw + 32 * half + 8 * c;  // first of 8 columns
        const uint4 val = make_uint4(pack_f16(v[8 * c], v[8 * c + 1]), pack_f16(v[8 * c + 2], v[8 * c + 3]),
                                     pack_f16(v[8 * c + 4], v[8 * c + 5]), pack_f16(v[8 * c + 6], v[8 * c + 7]));
        if (isW)
          *reinterpret_cast<uint4*>(ws + kSlotA1 + kmaj_off(64 + i, col, 128)) = val;
        else
          *reinterpret_cast<uint4*>(ws + kSlotU + (col >> 5) * 4096 + utile_off(i, col & 31)) = val;
      }
    }
  }
  tc_fence_before();
  cur = nxt;
  }
  if (gave_up) {  // let this CTA's last copies and products land (bounded) before it exits
    mbar_wait_bounded(bar_qk, (uint32_t)((it - 1) & 1));
    mbar_wait_bounded(bar_gv, (uint32_t)((it - 1) & 1));
    if (mma_count > 0) mbar_wait_bounded(bar_mma, (mma_count - 1) & 1u);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(kTmemCols));
}

template <int kGate, bool kL2>
static void launch_variant(const ChunkParams& p, unsigned grid, int64_t items, const ChunkMaps& maps,
                           cudaStream_t stream) {
  kda_chunk_kernel<kGate, kL2><<<grid, 256, kChunkSmem, stream>>>(p, items, maps);
}

namespace {
// cuTensorMapEncodeTiled, looked up once through the runtime (no link against
// the driver library)
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}
// [rows, H, 128] bf16 at `base` (rows of H * 256 bytes), 64 x 64 boxes
bool encode_input_map(CUtensorMap* m, const void* base, int64_t H, int64_t rows) {
  const EncodeTiled fn = encoder();
  if (!fn || rows < 1 || rows > INT32_MAX) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)(H * kHeadDim * 2)};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunk};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool launch_chunk_kernel(const ChunkParams& p, int64_t num_slots, cudaStream_t stream) {
  // the rows the kernel may touch from the row pointers: every sequence's
  // range (dense), or the packed tokens
  const int64_t rows = p.cu ? p.T : (p.N - 1) * p.ld + p.T;
  ChunkMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!encode_input_map(&maps.q, p.q, p.H, rows) || !encode_input_map(&maps.k, p.k, p.H, rows) ||
      !encode_input_map(&maps.v, p.v, p.H, rows) || (!p.g32 && !encode_input_map(&maps.g, p.g, p.H, rows)))
    return false;
  // persistent grid: two CTAs per SM (shared memory, registers and tensor-memory
  // columns all allow two), or fewer items
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t items = num_slots * p.H;
  const unsigned grid = (unsigned)min(items, (int64_t)(2 * (sms > 0 ? sms : 1)));
  const bool l2 = p.l2norm != 0;
  switch (p.gate_mode) {
    case kGateUnsafe:
      if (l2) launch_variant<kGateUnsafe, true>(p, grid, items, maps, stream);
      else launch_variant<kGateUnsafe, false>(p, grid, items, maps, stream);
      break;
    case kGateLogspace:
      if (l2) launch_variant<kGateLogspace, true>(p, grid, items, maps, stream);
      else launch_variant<kGateLogspace, false>(p, grid, items, maps, stream);
      break;
    default:
      if (l2) launch_variant<kGateSafe, true>(p, grid, items, maps, stream);
      else launch_variant<kGateSafe, false>(p, grid, items, maps, stream);
  }
  return true;
}

cudaError_t prepare_chunk_kernel() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const void* fns[] = {(const void*)kda_chunk_kernel<kGateSafe, true>,
                       (const void*)kda_chunk_kernel<kGateSafe, false>,
                       (const void*)kda_chunk_kernel<kGateUnsafe, true>,
                       (const void*)kda_chunk_kernel<kGateUnsafe, false>,
                       (const void*)kda_chunk_kernel<kGateLogspace, true>,
                       (const void*)kda_chunk_kernel<kGateLogspace, false>};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, attr, kChunkSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kda
