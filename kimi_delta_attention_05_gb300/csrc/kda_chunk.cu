// Intra-chunk stage of the KDA forward pass: one CTA per (64-token chunk, head).
//
// Computes, for its chunk, everything that does not depend on the recurrent
// state and stores it in the workspace slot of (chunk, head):
//   * the gate activation and the in-chunk cumulative decay (the "gate.py"
//     stage of the fla-kda code map: gate activation + cumulative decay),
//   * optional q/k L2 normalisation,
//   * A (beta-scaled strictly-lower decayed K K^T) and P (lower decayed Q K^T)
//     from 16-token sub-chunks: diagonal sub-blocks use an offset at the
//     sub-chunk midpoint, off-diagonal sub-blocks paired decay factors that
//     are both <= 1 (fla-kda SKILL.md, "Numerical invariants"; fla-kda skill
//     page on the midpoint offset),
//   * [W | U] = (I + A)^-1 Diag(beta) [K gamma | V] by block forward
//     substitution over the four sub-chunks: 16x16 diagonal inverses X_r by
//     forward substitution, M_rc = -X_r A_rc, then Y_r = X_r B_r + sum_{c<r} M_rc Y_c
//     (the "solve_tril" triangular block merges and the "wy_fast" WY
//     recompute of the fla-kda code map, fused),
//   * q gamma, k gamma_C / gamma and gamma_C for the state stage.
//
// Decay factors inside a sub-chunk come from running products of
// d_t = exp(a_t), so every exponent is taken once per (token, channel).
// The A and P operands are stored relative to the cumulative decay at the
// sub-chunk midpoint (after its 8th token); off-diagonal sub-blocks multiply
// in per-channel factors that move each side to the end of the earlier
// sub-chunk.  For these operands d_t is clamped below at exp(-10), so that the
// midpoint-relative values stay within [e^-80, e^80] for any gate; with the
// safe gate (a_t >= -5) the clamp never acts.  Where it acts, the true pair
// factor and the clamped one are both below exp(-10).  The recurrent-state
// quantities (q gamma, K gamma, k gamma_C / gamma, gamma_C) use the exact d_t.
//
// Precision: the A / P operands are bf16 (they need its exponent range); the
// diagonal inverses are fp32; everything else is fp16 (11-bit significand)
// with fp32 accumulation.
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime's entry-point query)

#include <cstring>
#include <mutex>

#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

// Tensor maps of the bf16 inputs [rows, H, 128]: 64 x 64 boxes (64 rows of one
// head, 64 channels) with the 128-byte swizzle, rows past the view zero-filled.
struct ChunkMaps {
  CUtensorMap q, k, v, g;
};

// exp(-10): floor of the per-token decay inside the A / P operands.
constexpr float kDiagDecayFloor = 4.5399929762484854e-05f;

// ---- shared-memory map (bytes) ----
// A "tile128" is 64 rows x 128 16-bit columns in two 8 KB halves, addressed by
// swz128 (the tensor-copy image of two 64 x 64 boxes with the 128-byte swizzle).
// phase 1 (until the A / P products are done)
constexpr int kCsQ = 0;          // tile128: raw q, then bf16 q_hat * xr
constexpr int kCsK = 16384;      // tile128: raw k, then bf16 k_hat * xr
constexpr int kCsKy = 32768;     // tile128: bf16 k_hat * yr
constexpr int kCsG = 49152;      // tile128: raw g, then fp16 beta k_hat gamma, then W
constexpr int kCsV = 65536;      // tile128: raw v
// phase 2 (in the raw v tile, dead once the operand pass has read it)
constexpr int kCsA16 = kCsV;            // tile64 fp16: A (lower sub-blocks)
constexpr int kCsAd = kCsV + 8192;      // fp32 [4][16][16]: diagonal sub-blocks of A
constexpr int kCsX = kCsV + 12288;      // tile64 fp16 [16][64]: inverse of sub-block r at cols 16r..
// small arrays
constexpr int kCsD = 81920;      // fp32 [8][128]: exact decay products of the 8-token half sub-chunks
constexpr int kCsXm = 86016;     // fp32 [4][128]: clamped product over tokens 0..7 of a sub-chunk
constexpr int kCsYm = 88064;     // fp32 [4][128]: clamped product over tokens 8..15
constexpr int kCsFa = 90112;     // bf16x2 [6][64]: left factors of the off-diagonal sub-blocks
constexpr int kCsYp = 91648;     // bf16x2 [4][64]: right factors (clamped product over tokens 8..15)
// Packed factor pairs are stored so that the pairs a K step of one mma fragment
// needs (channels ch, ch+1 and ch+8, ch+9, ch = 16 kk + 2 q4) are adjacent.
constexpr int kCsBeta = 93184;   // fp32 [64]
constexpr int kCsRq = 93440;     // fp32 [64]: 1 / |q| (or 1)
constexpr int kCsRk = 93696;     // fp32 [64]: 1 / |k| (or 1)
constexpr int kCsVt = 93952;     // tile128 [64 t][128 v] fp16: beta V, then U
constexpr int kCsBar = kCsVt + 16384;  // two mbarriers: q/k/g tiles, v tile
constexpr int kChunkSmem = kCsBar + 16;
static_assert(kCsQ % 1024 == 0 && kCsK % 1024 == 0 && kCsKy % 1024 == 0 && kCsG % 1024 == 0 &&
                  kCsV % 1024 == 0,
              "tensor-copy destinations with the 128-byte swizzle need 1024-byte alignment");

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Position of channel pair pp (channels 2 pp, 2 pp + 1) in a packed factor row.
__device__ __forceinline__ int fpair_pos(int pp) {
  return (pp & ~7) + 2 * (pp & 3) + ((pp >> 2) & 1);
}

__device__ __forceinline__ uint32_t& u32_at(unsigned char* base, uint32_t off) {
  return *reinterpret_cast<uint32_t*>(base + off);
}

// Packed bf16x2 multiply (fp32 exponent range, so a factor that underflows
// does so only where the scaled value is below ~1e-38 anyway).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Scale an A fragment (columns ch, ch+1 | ch+8, ch+9) by packed factors
// f01 = (f[ch], f[ch+1]), f89 = (f[ch+8], f[ch+9]).
__device__ __forceinline__ void scale_afrag(uint32_t (&a)[4], uint32_t f01, uint32_t f89) {
  a[0] = mul_bf16x2(a[0], f01);
  a[1] = mul_bf16x2(a[1], f01);
  a[2] = mul_bf16x2(a[2], f89);
  a[3] = mul_bf16x2(a[3], f89);
}
// Scale a B fragment pair (rows k = ch, ch+1 | ch+8, ch+9) likewise.
__device__ __forceinline__ void scale_bfrag(uint32_t& b0, uint32_t& b1, uint32_t f01, uint32_t f89) {
  b0 = mul_bf16x2(b0, f01);
  b1 = mul_bf16x2(b1, f89);
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

template <int kGate, bool kL2>
__global__ void __launch_bounds__(256, 2)
    kda_chunk_kernel(ChunkParams p, int64_t num_items, const __grid_constant__ ChunkMaps maps) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t H = p.H;
  const uint32_t sbase = smem_u32(smem);
  // Persistent: CTA b takes items b, b + gridDim.x, ... (item = slot * H + head).
  // The next item's q, k, g are copied in as soon as the A / P stage has finished
  // with the q, k and K yr tiles, and its v once the substitution is done with
  // the A / inverse tiles, so the copies overlap the rest of the current item.
  // Each tile is two tensor copies issued by one thread onto an mbarrier.
  if (p.cu) num_items = p.chunk_off[p.N] * H;  // varlen: only the slots in use
  struct Item {
    int64_t slot, t0;
    int h, L;
  };
  // ---- locate a chunk: sequence n, chunk i, first token t0, length L ----
  // (32-bit divisions whenever the item count allows: 64-bit ones are long
  // instruction sequences, run by every thread once per item)
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
  const uint32_t bar_qkg = sbase + kCsBar, bar_v = sbase + kCsBar + 8;
  // one thread: the q, k (and bf16 g) tiles of an item, two 64-column boxes each
  auto copy_qkg = [&](const Item& it, int gdst) {
    fence_proxy_async_smem();  // the tiles were last read by the generic proxy
    mbar_expect_tx(bar_qkg, (p.g32 ? 2u : 3u) * 16384u);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      tma_load_3d(sbase + kCsQ + hh * 8192, &maps.q, 64 * hh, it.h, (int)it.t0, bar_qkg);
      tma_load_3d(sbase + kCsK + hh * 8192, &maps.k, 64 * hh, it.h, (int)it.t0, bar_qkg);
      if (!p.g32) tma_load_3d(sbase + gdst + hh * 8192, &maps.g, 64 * hh, it.h, (int)it.t0, bar_qkg);
    }
  };
  auto copy_v = [&](const Item& it) {
    fence_proxy_async_smem();
    mbar_expect_tx(bar_v, 16384u);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      tma_load_3d(sbase + kCsV + hh * 8192, &maps.v, 64 * hh, it.h, (int)it.t0, bar_v);
  };
  // every thread: bounded wait for a tile phase; a wait that gives up sets the
  // status word, and the item goes on with whatever the tiles hold
  bool gave_up = false;
  auto wait_tiles = [&](uint32_t bar, uint32_t parity) {
    if (!gave_up && !mbar_wait_bounded(bar, parity)) {
      gave_up = true;
      atomicExch(p.status, 13);
    }
  };
  // rows L..63 of a tile copied past a short chunk's end (the next sequence's
  // rows, or zeros past the view) are cleared: the stages below expect zeros
  auto zero_tail = [&](int tile, int L) {
    for (int idx = tid; idx < (kChunk - L) * 16; idx += 256)
      *reinterpret_cast<uint4*>(smem + tile + swz128(L + (idx >> 4), 8 * (idx & 15))) =
          make_uint4(0u, 0u, 0u, 0u);
  };
  // beta input (logit, or beta itself) of token tid; 0 past the chunk end
  auto load_beta = [&](const Item& it) {
    return tid < it.L ? bf16_to_f(p.beta[(it.t0 + tid) * H + it.h]) : 0.f;
  };
  int64_t item = blockIdx.x;
  if (item >= num_items) return;
  Item cur = locate(item);
  if (tid == 0) {
    mbar_init(bar_qkg, 1);
    mbar_init(bar_v, 1);
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  __syncthreads();
  // The second CTA on each SM starts about a quarter of an item later, so that
  // the two CTAs sharing an SM run different stages (gate and operands on the
  // SFU / ALU pipes, products on the tensor cores) rather than the same ones
  // (T=8192 H=32: 155.9 -> 154.1 us; a 2.3 k or 9.2 k cycle offset 154.6 / 153.2).
  if (blockIdx.x >= (unsigned)p.second_wave) {
    const long long t0 = clock64();
    while (clock64() - t0 < 4600) __nanosleep(200);
  }
  // ---- S0 (first item only; later items were prefetched): q, k, g | v ----
  // (fp32 g is read in the gate stage itself)
  if (tid == 0) {
    copy_qkg(cur, kCsG);
    copy_v(cur);
  }
  float blogit = tid < kChunk ? load_beta(cur) : 0.f;
  float* sBeta = reinterpret_cast<float*>(smem + kCsBeta);

  int it = 0;
  for (; item < num_items; item += gridDim.x, ++it) {
  const int L = cur.L;
  const int h = cur.h;
  unsigned char* ws = p.ws + (cur.slot * H + h) * (int64_t)kSlotBytes;
  const int gt = (it & 1) ? kCsKy : kCsG;  // raw g, then beta K gamma, then W
  const int yt = (it & 1) ? kCsG : kCsKy;  // bf16 K yr
  const int64_t next = item + gridDim.x;
  Item nxt = cur;
  if (next < num_items) nxt = locate(next);
  if (tid < kChunk)
    sBeta[tid] = tid >= L ? 0.f : (p.beta_prob ? blogit : rcp_approx(1.0f + ex2(-blogit * kLog2e)));
  wait_tiles(bar_qkg, (uint32_t)(it & 1));  // q, k, g of this item (v may still be in flight)
  if (L < kChunk) {
    zero_tail(kCsQ, L);
    zero_tail(kCsK, L);
    if (!p.g32) zero_tail(gt, L);
  }
  __syncthreads();

  // ---- S1: per-token inverse norms of q and k (two threads per row, 64 channels each) ----
  float* sRq = reinterpret_cast<float*>(smem + kCsRq);
  float* sRk = reinterpret_cast<float*>(smem + kCsRk);
  {
    const int row = tid >> 1, half = tid & 1;  // rows 0..63 of q, 64..127 of k
    const int t = row & 63;
    float ss = 0.f;
    if (kL2) {
      const unsigned char* tile = smem + (row < 64 ? kCsQ : kCsK);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(tile + half * 8192 + t * 128 + ((c ^ (t & 7)) << 4));
        const float2 a = unpack_bf16(v.x), b = unpack_bf16(v.y), e = unpack_bf16(v.z), f = unpack_bf16(v.w);
        ss += a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y + e.x * e.x + e.y * e.y + f.x * f.x + f.y * f.y;
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    }
    if (half == 0) (row < 64 ? sRq : sRk)[t] = kL2 ? rsqrtf(ss + 1e-6f) : 1.0f;
  }

  // ---- S2: gate activation, per-token decays d (registers), half sub-chunk products ----
  // thread -> sub-chunk rb, half hf (tokens 8 hf .. 8 hf + 7 of it), channels c0 .. c0 + 3;
  // a warp covers all 128 channels of one half, so every token row is one access
  const int cg = tid & 31, hf = (tid >> 5) & 1, rb = tid >> 6;
  const int c0 = 4 * cg;
  const int seg = 2 * rb + hf;      // half sub-chunk index 0..7
  const int tb = 16 * rb + 8 * hf;  // its first token
  float* sD = reinterpret_cast<float*>(smem + kCsD);
  float* sXm = reinterpret_cast<float*>(smem + kCsXm);
  float* sYm = reinterpret_cast<float*>(smem + kCsYm);
  float* sFa = reinterpret_cast<float*>(smem + kCsFa);
  // decays of channel pairs (c0, c0 + 1), (c0 + 2, c0 + 3) in f32x2 registers
  f32x2 d2[8][2];
  float inv[4];  // 1 / (clamped product over this half)
  const f32x2 one2 = f2(1.0f, 1.0f);
  {
    const float4 dtb = (p.dt_bias && kGate != kGateLogspace)
                           ? *reinterpret_cast<const float4*>(p.dt_bias + h * kHeadDim + c0)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    const f32x2 dtb2[2] = {f2(dtb.x, dtb.y), f2(dtb.z, dtb.w)};
    const float amul_log2e = (p.A_log && kGate != kGateLogspace ? expf(p.A_log[h]) : 1.0f) *
                             (kGate == kGateUnsafe ? 1.0f : kLog2e);
    const float lb_log2e = p.lower_bound * kLog2e;
    f32x2 D2[2] = {one2, one2}, Dc2[2] = {one2, one2};
    // decay of token tb + j from its gate input pair values
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
        const uint2 graw = *reinterpret_cast<const uint2*>(smem + gt + swz128(tb + j, c0));
        gate_token(j, bf2_to_f2(graw.x), bf2_to_f2(graw.y));
      }
    }
    const float2 Da = f2u(D2[0]), Db = f2u(D2[1]), Dca = f2u(Dc2[0]), Dcb = f2u(Dc2[1]);
    *reinterpret_cast<float4*>(sD + seg * 128 + c0) = make_float4(Da.x, Da.y, Db.x, Db.y);
    *reinterpret_cast<float4*>((hf ? sYm : sXm) + rb * 128 + c0) = make_float4(Dca.x, Dca.y, Dcb.x, Dcb.y);
    if (hf) {
      uint32_t* yp = reinterpret_cast<uint32_t*>(smem + kCsYp) + rb * 64;
      yp[fpair_pos(2 * cg)] = pack_bf16(Dca.x, Dca.y);
      yp[fpair_pos(2 * cg + 1)] = pack_bf16(Dcb.x, Dcb.y);
    }
    inv[0] = __frcp_rn(Dca.x);
    inv[1] = __frcp_rn(Dca.y);
    inv[2] = __frcp_rn(Dcb.x);
    inv[3] = __frcp_rn(Dcb.y);
  }
  __syncthreads();

  // ---- S3: operands (same thread mapping) ----
  //  exact, chunk relative:     gamma_j = prod_{s<=j} d_s  -> beta K gamma (smem), q gamma (ws)
  //  exact, chunk-end relative: gamma_C / gamma_j           -> k_hat (ws)
  //  clamped, midpoint relative: xr_j = e^{lam_j - lam_7}, yr_j = 1 / xr_j -> A / P operands;
  //  within the half before the midpoint xr_j = inv * (clamped product up to j), after
  //  it xr_j = clamped product from token 8 up to j, so each half needs only its own d
  {
    f32x2 pre2[2] = {one2, one2}, suf2[2] = {one2, one2};
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) {
      const float4 Ds = *reinterpret_cast<const float4*>(sD + s2 * 128 + c0);
      const f32x2 dv2[2] = {f2(Ds.x, Ds.y), f2(Ds.z, Ds.w)};
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        if (s2 < seg) pre2[pp] = mul2(pre2[pp], dv2[pp]);
        if (s2 > seg) suf2[pp] = mul2(suf2[pp], dv2[pp]);
      }
    }
    if (tid < 32) {  // left factors of the off-diagonal sub-blocks (r, cb), cb < r
#pragma unroll
      for (int r = 1; r < 4; ++r)
#pragma unroll
        for (int cb = 0; cb < r; ++cb) {
          float4 e = *reinterpret_cast<const float4*>(sXm + r * 128 + c0);
          for (int s3 = cb + 1; s3 < r; ++s3) {
            const float4 xm = *reinterpret_cast<const float4*>(sXm + s3 * 128 + c0);
            const float4 ym = *reinterpret_cast<const float4*>(sYm + s3 * 128 + c0);
            e.x *= xm.x * ym.x;
            e.y *= xm.y * ym.y;
            e.z *= xm.z * ym.z;
            e.w *= xm.w * ym.w;
          }
          uint32_t* fp = reinterpret_cast<uint32_t*>(sFa) + (r * (r - 1) / 2 + cb) * 64;
          fp[fpair_pos(2 * cg)] = pack_bf16(e.x, e.y);
          fp[fpair_pos(2 * cg + 1)] = pack_bf16(e.z, e.w);
        }
      // gamma_C = product over all eight halves
      const float2 sa = f2u(suf2[0]), sb = f2u(suf2[1]);
      *reinterpret_cast<float4*>(ws + kSlotGc + c0 * 4) =
          make_float4(sa.x * sD[c0], sa.y * sD[c0 + 1], sb.x * sD[c0 + 2], sb.y * sD[c0 + 3]);
    }
    // xr takes 1 / (clamped product) in the first half, yr in the second
    const f32x2 invx2[2] = {hf ? one2 : f2(inv[0], inv[1]), hf ? one2 : f2(inv[2], inv[3])};
    const f32x2 inv2[2] = {hf ? f2(inv[0], inv[1]) : one2, hf ? f2(inv[2], inv[3]) : one2};
    unsigned char* gQg = ws + kSlotA1;  // rows 0..63 of the [q gamma; W] image
    unsigned char* gKh = ws + kSlotKh;
    // backward over the half (reads the raw k)
    {
      f32x2 y2[2] = {suf2[0], suf2[1]}, yc2[2] = {one2, one2};
#pragma unroll
      for (int j = 7; j >= 0; --j) {
        const int t = tb + j;
        const uint32_t off = swz128(t, c0);
        const float rk = sRk[t];
        const f32x2 rk2 = f2(rk, rk);
        const uint2 kraw = *reinterpret_cast<const uint2*>(smem + kCsK + off);
        const f32x2 k2[2] = {mul2(bf2_to_f2(kraw.x), rk2), mul2(bf2_to_f2(kraw.y), rk2)};
        const f32x2 yr2[2] = {mul2(yc2[0], inv2[0]), mul2(yc2[1], inv2[1])};  // inv = 1 in the first half
        *reinterpret_cast<uint2*>(smem + yt + off) =
            make_uint2(pack_bf16_2(mul2(k2[0], yr2[0])), pack_bf16_2(mul2(k2[1], yr2[1])));
        *reinterpret_cast<uint2*>(gKh + kmaj_off(t, c0, 64)) =
            make_uint2(pack_f16_2(mul2(k2[0], y2[0])), pack_f16_2(mul2(k2[1], y2[1])));
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          y2[pp] = mul2(y2[pp], d2[j][pp]);
          yc2[pp] = mul2(yc2[pp], max2_floor(d2[j][pp]));
        }
      }
    }
    wait_tiles(bar_v, (uint32_t)(it & 1));  // v of this item
    if (L < kChunk) zero_tail(kCsV, L);
    __syncthreads();
    // forward over the half (overwrites raw q, k, g, v)
    {
      f32x2 x2[2] = {pre2[0], pre2[1]}, xc2[2] = {one2, one2};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int t = tb + j;
        const uint32_t off = swz128(t, c0);
        f32x2 xr2[2];
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          x2[pp] = mul2(x2[pp], d2[j][pp]);
          xc2[pp] = mul2(xc2[pp], max2_floor(d2[j][pp]));
          xr2[pp] = mul2(xc2[pp], invx2[pp]);  // invx = 1 in the second half
        }
        const float rk = sRk[t], rq = sRq[t], bt = sBeta[t];
        const f32x2 rk2 = f2(rk, rk), rq2 = f2(rq, rq), bt2 = f2(bt, bt);
        const uint2 kraw = *reinterpret_cast<const uint2*>(smem + kCsK + off);
        const uint2 qraw = *reinterpret_cast<const uint2*>(smem + kCsQ + off);
        const uint2 vraw = *reinterpret_cast<const uint2*>(smem + kCsV + off);
        const f32x2 k2[2] = {mul2(bf2_to_f2(kraw.x), rk2), mul2(bf2_to_f2(kraw.y), rk2)};
        const f32x2 q2[2] = {mul2(bf2_to_f2(qraw.x), rq2), mul2(bf2_to_f2(qraw.y), rq2)};
        const f32x2 v2[2] = {bf2_to_f2(vraw.x), bf2_to_f2(vraw.y)};
        *reinterpret_cast<uint2*>(smem + kCsK + off) =
            make_uint2(pack_bf16_2(mul2(k2[0], xr2[0])), pack_bf16_2(mul2(k2[1], xr2[1])));
        *reinterpret_cast<uint2*>(smem + kCsQ + off) =
            make_uint2(pack_bf16_2(mul2(q2[0], xr2[0])), pack_bf16_2(mul2(q2[1], xr2[1])));
        *reinterpret_cast<uint2*>(smem + gt + off) =
            make_uint2(pack_f16_2(mul2(mul2(bt2, k2[0]), x2[0])), pack_f16_2(mul2(mul2(bt2, k2[1]), x2[1])));
        *reinterpret_cast<uint2*>(smem + kCsVt + off) =
            make_uint2(pack_f16_2(mul2(bt2, v2[0])), pack_f16_2(mul2(bt2, v2[1])));
        *reinterpret_cast<uint2*>(gQg + kmaj_off(t, c0, 128)) =
            make_uint2(pack_f16_2(mul2(q2[0], x2[0])), pack_f16_2(mul2(q2[1], x2[1])));
      }
    }
  }
  __syncthreads();

  // ---- S4: A (beta-scaled strictly lower decayed K K^T: fp16 operand tile plus fp32
  //      diagonal sub-blocks) and P (lower decayed Q K^T, into the workspace), per
  //      sub-block pair (r, cb <= r).  One warp computes A and P of a pair together:
  //      the K yr fragment and its factor are shared, and the K xr and Q xr fragments
  //      take the same left factor.  Warps 0-5: the off-diagonal pairs
  //      (1,0) (2,0) (2,1) (3,0) (3,1) (3,2); warps 6, 7: two diagonal pairs each.
  const int g = lane >> 2, q4 = lane & 3;
  float* sAd = reinterpret_cast<float*>(smem + kCsAd);
  {
    unsigned char* gP = ws + kSlotP;  // kmaj image R=64, K=64
    const uint32_t* fap = reinterpret_cast<const uint32_t*>(sFa);
    const uint32_t* ybp = reinterpret_cast<const uint32_t*>(smem + kCsYp);
    auto epilogue = [&](int mat, int r, int cb, const float (&acc)[2][4]) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = 16 * r + g + 8 * hh;
          const int col = 16 * cb + 8 * nt + 2 * q4;
          const float v0 = acc[nt][2 * hh], v1 = acc[nt][2 * hh + 1];
          if (mat == 0) {
            const float bt = sBeta[row];
            const float a0 = (cb < r || col < row) ? v0 * bt : 0.f;
            const float a1 = (cb < r || col + 1 < row) ? v1 * bt : 0.f;
            u32_at(smem + kCsA16, swz64(row, col)) = pack_f16(a0, a1);
            if (cb == r)
              *reinterpret_cast<float2*>(sAd + r * 256 + (row - 16 * r) * 16 + (col - 16 * r)) =
                  make_float2(a0, a1);
          } else {
            const bool k0 = cb < r || col <= row;
            const bool k1 = cb < r || col + 1 <= row;
            u32_at(gP, kmaj_off(row, col, 64)) = pack_f16(k0 ? v0 : 0.f, k1 ? v1 : 0.f);
          }
        }
      }
    };
#pragma unroll 1
    for (int task = 0; task < (warp < 6 ? 1 : 2); ++task) {
      int r, cb;
      if (warp < 6) {
        r = warp < 1 ? 1 : (warp < 3 ? 2 : 3);
        cb = warp - r * (r - 1) / 2;
      } else {
        r = cb = (warp - 6) + 2 * task;
      }
      float accA[2][4], accP[2][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) accA[a][e] = accP[a][e] = 0.f;
      if (cb < r) {
        const uint32_t* fa = fap + (r * (r - 1) / 2 + cb) * 64 + 2 * q4;
        const uint32_t* fb = ybp + cb * 64 + 2 * q4;
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t ak[4], aq[4], b[4];
          lda_128(ak, sbase + kCsK, 16 * r, 16 * kk, lane);
          lda_128(aq, sbase + kCsQ, 16 * r, 16 * kk, lane);
          ldb_nk_128(b, sbase + yt, 16 * cb, 16 * kk, lane);
          const uint2 pa = *reinterpret_cast<const uint2*>(fa + 8 * kk);
          const uint2 pb = *reinterpret_cast<const uint2*>(fb + 8 * kk);
          scale_afrag(ak, pa.x, pa.y);
          scale_afrag(aq, pa.x, pa.y);
          scale_bfrag(b[0], b[1], pb.x, pb.y);
          scale_bfrag(b[2], b[3], pb.x, pb.y);
          mma_bf16(accA[0], ak, b[0], b[1]);
          mma_bf16(accA[1], ak, b[2], b[3]);
          mma_bf16(accP[0], aq, b[0], b[1]);
          mma_bf16(accP[1], aq, b[2], b[3]);
        }
      } else {
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t ak[4], aq[4], b[4];
          lda_128(ak, sbase + kCsK, 16 * r, 16 * kk, lane);
          lda_128(aq, sbase + kCsQ, 16 * r, 16 * kk, lane);
          ldb_nk_128(b, sbase + yt, 16 * cb, 16 * kk, lane);
          mma_bf16(accA[0], ak, b[0], b[1]);
          mma_bf16(accA[1], ak, b[2], b[3]);
          mma_bf16(accP[0], aq, b[0], b[1]);
          mma_bf16(accP[1], aq, b[2], b[3]);
        }
      }
      epilogue(0, r, cb, accA);
      epilogue(1, r, cb, accP);
    }
    // tiles above the diagonal: zero in A (read by the substitution) and in P
    for (int idx = tid; idx < 6 * 128; idx += 256) {
      const int o = idx >> 7, e = idx & 127;  // upper sub-block pairs (r, cb), cb > r
      const int r = o < 3 ? 0 : (o < 5 ? 1 : 2);
      const int cb = r + 1 + (o - (r == 0 ? 0 : (r == 1 ? 3 : 5)));
      const int row = 16 * r + (e >> 3), col = 16 * cb + 2 * (e & 7);
      u32_at(smem + kCsA16, swz64(row, col)) = 0u;
      u32_at(gP, kmaj_off(row, col, 64)) = 0u;
    }
  }
  __syncthreads();
  // q, k, K yr tiles are free: next item's q, k, g (g into this item's K yr tile)
  if (next < num_items) {
    if (tid == 128) copy_qkg(nxt, yt);  // warp 4: idle in the substitution below
    if (tid < kChunk) blogit = load_beta(nxt);
  }

  // ---- S6: X_r = (I + A_rr)^-1 by forward substitution (warp r, lane = column) ----
  if (warp < 4 && lane < 16) {
    const int j = lane;
    const float4* Ad4 = reinterpret_cast<const float4*>(sAd + warp * 256);  // rows of 16 floats
    float x[kSub];
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii) {
      float acc = 0.f;
#pragma unroll
      for (int s4 = 0; 4 * s4 < ii; ++s4) {  // row ii, four entries per 16-byte load
        const float4 a = Ad4[ii * 4 + s4];
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (4 * s4 + c < ii) acc += av[c] * x[4 * s4 + c];
      }
      x[ii] = (ii == j) ? 1.f : (ii < j ? 0.f : -acc);
    }
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii)
      *reinterpret_cast<__half*>(smem + kCsX + swz64(ii, 16 * warp + j)) = __float2half_rn(x[ii]);
  }
  __syncthreads();

  // ---- S6b: M_rc = -X_r A_rc for the off-diagonal sub-blocks c < r (warp w < 6 takes
  //      pair w in the order (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)), written over A_rc ----
  if (warp < 6) {
    const int r = warp < 1 ? 1 : (warp < 3 ? 2 : 3);
    const int c = warp - r * (r - 1) / 2;
    float acc[2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
    uint32_t a[4], b[4];
    lda_64(a, sbase + kCsX, 0, 16 * r, lane);
    ldb_kn_64(b, sbase + kCsA16, 16 * c, 16 * r, lane);
    mma_f16(acc[0], a, b[0], b[1]);
    mma_f16(acc[1], a, b[2], b[3]);
    __syncwarp();
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
        u32_at(smem + kCsA16, swz64(16 * r + g + 8 * hh, 16 * c + 8 * nt + 2 * q4)) =
            pack_f16(-acc[nt][2 * hh], -acc[nt][2 * hh + 1]);
  }
  __syncthreads();

  // ---- S7: [W | U] rows of sub-chunk r: Y_r = X_r B_r + sum_{c<r} M_rc Y_c, accumulated
  //      in registers and written over B_r; warp -> 32 columns of B = [beta K gamma | beta V]
  //      (warp-private: only __syncwarp) ----
  {
    const int cbase = 32 * (warp & 3);
    unsigned char* buf = smem + (warp < 4 ? gt : kCsVt);
    const uint32_t bufa = sbase + (warp < 4 ? gt : kCsVt);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float y[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) y[a][e] = 0.f;
#pragma unroll
      for (int c = 0; c <= r; ++c) {
        uint32_t a[4];
        if (c == r) lda_64(a, sbase + kCsX, 0, 16 * r, lane);
        else lda_64(a, sbase + kCsA16, 16 * r, 16 * c, lane);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b[4];
          ldb_kn_128(b, bufa, cbase + 16 * np, 16 * c, lane);
          mma_f16(y[2 * np], a, b[0], b[1]);
          mma_f16(y[2 * np + 1], a, b[2], b[3]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t off = swz128(16 * r + g + 8 * hh, cbase + 8 * nt + 2 * q4);
          u32_at(buf, off) = pack_f16(y[nt][2 * hh], y[nt][2 * hh + 1]);
        }
      __syncwarp();
    }
  }
  fence_proxy_async_smem();  // W (rows of gt) is read next by bulk copies
  __syncthreads();
  // the A / inverse tiles in the raw-v tile are free: next item's v
  if (next < num_items && tid == 0) copy_v(nxt);
  // W: each 64-column half of the tile is byte for byte the half of rows 64..127
  // of the [q gamma; W] image (same 128-byte rows, same row % 8 chunk order)
  if (tid == 32) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], 8192;\n" ::"l"(ws + kSlotA1 + hh * 16384 + 64 * 128),
                   "r"(sbase + gt + hh * 8192) : "memory");
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
  }

  // ---- S8: U into the four per-value-tile images, 16-byte chunks remapped from
  //      the tile128 layout (W went out above by bulk copies) ----
#pragma unroll 4
  for (int idx = tid; idx < 1024; idx += 256) {
    const int t = (idx >> 4) & 63, c = idx & 15;
    const uint4 val = *reinterpret_cast<const uint4*>(smem + kCsVt + swz128(t, 8 * c));
    *reinterpret_cast<uint4*>(ws + kSlotU + (c >> 2) * 4096 + utile_off(t, (c & 3) * 8)) = val;
  }
  if (tid == 32)  // the W copies have read gt before the next item writes it
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
  cur = nxt;
  }
  if (tid == 32)  // the W stores complete before the CTA exits
    asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
  if (gave_up) {  // let this CTA's last copies land (bounded) before it exits
    mbar_wait_bounded(bar_qkg, (uint32_t)((it - 1) & 1));
    mbar_wait_bounded(bar_v, (uint32_t)((it - 1) & 1));
  }
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

bool launch_chunk_kernel(const ChunkParams& p, int64_t num_slots, cudaStream_t stream,
                         int busy_sms) {
  // the rows the kernel may touch from the row pointers: every sequence's
  // range (dense), or the packed tokens
  const int64_t rows = p.cu ? p.T : (p.N - 1) * p.ld + p.T;
  ChunkMaps maps;
  memset(&maps, 0, sizeof(maps));
  if (!encode_input_map(&maps.q, p.q, p.H, rows) || !encode_input_map(&maps.k, p.k, p.H, rows) ||
      !encode_input_map(&maps.v, p.v, p.H, rows) || (!p.g32 && !encode_input_map(&maps.g, p.g, p.H, rows)))
    return false;
  // persistent grid: two CTAs per SM (the shared-memory and register budget) on
  // the SMs another kernel does not hold, or fewer items
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t items = num_slots * p.H;
  const int free_sms = sms - busy_sms > 0 ? sms - busy_sms : 1;
  const unsigned grid = (unsigned)min(items, (int64_t)(2 * free_sms));
  ChunkParams q = p;
  q.second_wave = grid == (unsigned)(2 * free_sms) ? free_sms : INT32_MAX;  // full two-per-SM grids only
  const bool l2 = p.l2norm != 0;
  switch (p.gate_mode) {
    case kGateUnsafe:
      if (l2) launch_variant<kGateUnsafe, true>(q, grid, items, maps, stream);
      else launch_variant<kGateUnsafe, false>(q, grid, items, maps, stream);
      break;
    case kGateLogspace:
      if (l2) launch_variant<kGateLogspace, true>(q, grid, items, maps, stream);
      else launch_variant<kGateLogspace, false>(q, grid, items, maps, stream);
      break;
    default:
      if (l2) launch_variant<kGateSafe, true>(q, grid, items, maps, stream);
      else launch_variant<kGateSafe, false>(q, grid, items, maps, stream);
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
