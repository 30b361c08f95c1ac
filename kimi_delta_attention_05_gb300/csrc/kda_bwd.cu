// Backward pass of the KDA forward in chunked (WY / UT) form, the "chunk_bwd"
// stage of the fla-kda code map: gradients of L = <out, dout> +
// <final_state, dfinal_state> with respect to q, k, v, g, beta, A_log, dt_bias
// and the initial state.  All arithmetic is fp32.
//
// Per (sequence, head) the tokens are cut into 64-token chunks; a chunk's rows
// t = 0..63 are padded past its length L with zero q, k, v, beta and gate.  With
// S the [V][K] state before the chunk and q, k L2-normalised if asked:
//   Gamma_t = sum_{s<=t} a_s                      in-chunk cumulative log decay
//   G_ts = sum_c k_tc k_sc e^{Gamma_tc - Gamma_sc}  (s < t)
//   P_ts = sum_c q_tc k_sc e^{Gamma_tc - Gamma_sc}  (s <= t)
//   M = I + Diag(beta) G,  Minv = M^-1,  T = Minv Diag(beta)
//   Qg = q e^Gamma,  Kg = k e^Gamma,  Khat = k e^{Gamma_C - Gamma},  gC = e^{Gamma_C}
//   W = T Kg,  U = T V,  Unew = U - W S^T
//   O = scale (Qg S^T + P Unew),  S_C = S Diag(gC) + Unew^T Khat
// (Gamma_C is the last row; the padded rows leave it equal to Gamma_{L-1}.)
// Reverse mode, with dO = dL/dO and dS_C = dL/dS_C:
//   dU   = scale P^T dO + Khat dS_C^T,   dS = scale dO^T Qg + dS_C Diag(gC) - dU^T W
//   dQg  = scale dO S,  dP = scale dO Unew^T,  dKhat = Unew dS_C,  dgC = colsum(S . dS_C)
//   dW   = -dU S,  dV = T^T dU,  dKg = T^T dW,  dT = dU V^T + dW Kg^T
//   dbeta_t = (Minv^T dT)_tt + sum_s dA_ts G_ts,  dM = -Minv^T (dT Diag(beta)) Minv^T,
//   dA = strict_lower(dM),  dG = Diag(beta) dA
// then through the pairwise products G, P, the e^Gamma scalings, the cumulative
// sum (da_s = sum_{t>=s} dGamma_t), the gate, the L2 norm and the sigmoid of beta.
// The pairwise factor e^{Gamma_t - Gamma_s} (s <= t) is never formed from
// exponentials of single rows (they can overflow): inside a 16-token block it is
// taken pair by pair, across blocks it splits at the first token r of t's block
// into e^{Gamma_t - Gamma_r} e^{Gamma_r - Gamma_s}, both factors at most 1.
//
// Launches:
//  1. prep, one CTA per (chunk, head): Gamma, G, P, Minv, W, U, Khat, Qg, Kg, gC
//     into the chunk's workspace item, with the normalised rows, beta, the norm
//     factors and the gate's derivatives for launch 5;
//  2. forward state pass, one CTA per (sequence, head, 32 value rows): walks the
//     chunks, storing S before each chunk and Unew (value rows are independent);
//  3. reverse state pass, same grid, chunks last to first from dfinal: stores
//     dS_C and dU of each chunk, then dinitial;
//  4. gradient products, one CTA per (chunk, head): dQg, dKhat, dKg, dP, dT, dgC, dv;
//  5. chunk gradients, one CTA per (chunk, head): dM, dG, dbeta, the pairwise
//     terms, the scalings, the cumulative sum, gate and norm derivatives: dq,
//     dk, dg, dbeta, and the chunk's parts of dA_log and dt_bias;
//  6. finalize, one CTA per head: those parts summed over the chunks in order.
#include <atomic>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

// Backward parameters.
struct BwdParams {
  const uint16_t *q, *k, *v, *g, *beta, *dout;  // bf16 inputs and dL/d out
  const float* g32;                             // g as fp32, or nullptr
  const float* A_log;
  const float* dt_bias;
  float lower_bound, scale;
  int gate_mode, beta_prob, l2norm;
  const void* init;                             // [N, H, 128, 128] or nullptr
  int init_bf16;
  const float* dfinal;                          // [N, H, 128, 128] fp32 or nullptr
  const int64_t* cu;                            // [N + 1] or nullptr (dense)
  const int64_t* chunk_off;                     // [N + 1] chunk prefix (varlen)
  int64_t N, T, H, NT;                          // NT: chunks per sequence (dense)
  int64_t nslots;                               // chunk slots; items = nslots * H
  float* ws;                                    // items of kItemFloats
  float *dq, *dk, *dv, *dg, *dbeta;             // fp32 gradients
  float *dA_log, *ddt_bias, *dinit;             // fp32, each may be nullptr
};

namespace {

constexpr int kC = kChunk;    // 64 tokens per chunk
constexpr int kD = kHeadDim;  // 128
constexpr int kLd = 132;      // row stride (floats) of [64][128] shared arrays (bank spread)
constexpr int kLs = 68;       // row stride of [64][64] shared arrays

// Workspace item of a (chunk slot, head), fp32 blocks (row-major):
constexpr int kItemW = 0;         // W [64][128]; dKg after the reverse pass
constexpr int kItemU = 8192;      // U [64][128]; Unew after the forward pass
constexpr int kItemKh = 16384;    // Khat [64][128]; dKhat after the reverse pass
constexpr int kItemQg = 24576;    // Qg [64][128]; dQg after the reverse pass
constexpr int kItemKg = 32768;    // Kg [64][128]
constexpr int kItemP = 40960;     // P [64][64] (lower incl. diagonal); dP after the reverse pass
constexpr int kItemMi = 45056;    // Minv [64][64]
constexpr int kItemG = 49152;     // G [64][64] (strictly lower)
constexpr int kItemS0 = 53248;    // S before the chunk [128 v][128 k]
constexpr int kItemDS = 69632;    // dS_C [128][128]
constexpr int kItemDU = 86016;    // dU [64][128]
constexpr int kItemDT = 94208;    // dT [64][64]
constexpr int kItemGC = 98304;    // gC [128]
constexpr int kItemDGC = 98432;   // dgC [128]
constexpr int kItemPart = 98560;  // parts of ddt_bias [128] and dA_log [1]
constexpr int kItemQh = 98752;    // q (L2-normalised if asked) [64][128]
constexpr int kItemKn = 106944;   // k (L2-normalised if asked) [64][128]
constexpr int kItemGm = 115136;   // Gamma [64][128]
constexpr int kItemDz = 123328;   // da/dz of the gate [64][128]
constexpr int kItemDa = 131520;   // da/dA_log of the gate [64][128]
constexpr int kItemVec = 139712;  // beta [64], norm factors of q [64] and k [64]
constexpr int kItemFloats = 139968;  // 559,872 bytes, a multiple of 256
static_assert(kItemPart + kD + 1 <= kItemQh && kItemVec + 3 * kC <= kItemFloats && kItemFloats % 64 == 0,
              "item layout");

constexpr int kStage = 16 * (kLs + kLd);  // GEMM staging floats
constexpr int kProdFloats = kC * kLd + kStage;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}
__device__ __forceinline__ void load4(const uint16_t* p, float (&x)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const float2 a = unpack_bf16(r.x), b = unpack_bf16(r.y);
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
// packed pairs of fp32 (low word = first element) and the paired FMA, two
// IEEE fused multiply-adds per instruction
typedef unsigned long long f2_t;
__device__ __forceinline__ f2_t pk2(float a, float b) {
  f2_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 up2(f2_t r) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
  return f;
}
__device__ __forceinline__ f2_t fma2(f2_t a, f2_t b, f2_t c) {
  f2_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ ulonglong2 ld2x2(const float* p) { return *reinterpret_cast<const ulonglong2*>(p); }
// e^x of a decay exponent (x <= 0 up to rounding): the fast exponential, whose
// error (a few ulp, growing with |x|) stays far inside the gradients'
// tolerance; the accurate expf gives the same gradient errors at full size
__device__ __forceinline__ float dexp(float x) { return __expf(x); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// Activated log decay a = gate(z) and its derivatives da/dz, da/dA_log
// (amul = exp(A_log), or 1 without A_log): safe lb sigmoid(amul z), unsafe
// -amul softplus(z), logspace z itself.
__device__ __forceinline__ float gate_a(int mode, float z, float amul, float lb, float& dadz,
                                        float& dadA) {
  if (mode == kGateLogspace) {
    dadz = 1.f;
    dadA = 0.f;
    return z;
  }
  if (mode == kGateUnsafe) {
    const float sp = fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));
    const float a = -amul * sp;
    dadz = -amul / (1.f + expf(-z));
    dadA = a;
    return a;
  }
  const float x = amul * z;
  const float s = 1.f / (1.f + expf(-x));
  const float ds = s * (1.f - s);
  dadz = lb * ds * amul;
  dadA = lb * ds * x;
  return lb * s;
}

__device__ __forceinline__ float gate_mul(const BwdParams& p, int h) {
  return (p.A_log && p.gate_mode != kGateLogspace) ? expf(p.A_log[h]) : 1.f;
}
// Token range of a chunk slot: rows t0 .. t0 + L - 1 of sequence n.  False for
// a slot past the last chunk (varlen workspaces are sized for the worst case).
struct ChunkLoc {
  int64_t t0, n;
  int L;
};
__device__ __forceinline__ bool locate(const BwdParams& p, int64_t slot, ChunkLoc& c) {
  if (!p.cu) {
    c.n = slot / p.NT;
    const int64_t ci = slot - c.n * p.NT;
    c.t0 = c.n * p.T + ci * kC;
    c.L = (int)min((int64_t)kC, p.T - ci * kC);
    return true;
  }
  if (slot >= p.chunk_off[p.N]) return false;
  int64_t lo = 0, hi = p.N - 1;  // largest n with chunk_off[n] <= slot
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (p.chunk_off[mid] <= slot) lo = mid;
    else hi = mid - 1;
  }
  c.n = lo;
  const int64_t ci = slot - p.chunk_off[lo];
  c.t0 = p.cu[lo] + ci * kC;
  c.L = (int)min((int64_t)kC, p.cu[lo + 1] - c.t0);
  return true;
}

// Chunk slots of sequence n: first and count.
__device__ __forceinline__ void seq_chunks(const BwdParams& p, int64_t n, int64_t& first, int64_t& count) {
  if (!p.cu) {
    first = n * p.NT;
    count = p.NT;
  } else {
    first = p.chunk_off[n];
    count = p.chunk_off[n + 1] - first;
  }
}

// The chunk's rows of k and q (L2-normalised if asked) into Kh, Qh [64][kLd],
// beta into vb, the norm factors 1 / sqrt(|x|^2 + eps) into rq, rk (if given);
// rows >= L are zero.  One warp per row, lane = 4 channels; kNT threads.
template <int kNT>
__device__ void load_rows(const BwdParams& p, const ChunkLoc& cl, int h, float* Kh, float* Qh,
                          float* vb, float* rq, float* rk) {
  constexpr int kNW = kNT / 32, kRows = kC / kNW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float q[kRows][4], k[kRows][4], braw[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {  // every load of the warp's rows before any use (rows
    const int t = min(warp + kNW * i, cl.L - 1);  // past the chunk re-read its last row)
    const int64_t row = (cl.t0 + t) * p.H + h;
    load4(p.q + row * kD + 4 * lane, q[i]);
    load4(p.k + row * kD + 4 * lane, k[i]);
    braw[i] = bf16_to_f(p.beta[row]);
  }
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int t = warp + kNW * i;
    if (t >= cl.L) {
#pragma unroll
      for (int c = 0; c < 4; ++c) q[i][c] = k[i][c] = 0.f;
    }
    float sq = 1.f, sk = 1.f;
    if (p.l2norm) {
      sq = rsqrtf(warp_sum(q[i][0] * q[i][0] + q[i][1] * q[i][1] + q[i][2] * q[i][2] + q[i][3] * q[i][3]) + 1e-6f);
      sk = rsqrtf(warp_sum(k[i][0] * k[i][0] + k[i][1] * k[i][1] + k[i][2] * k[i][2] + k[i][3] * k[i][3]) + 1e-6f);
    }
    st4(Qh + t * kLd + 4 * lane, q[i][0] * sq, q[i][1] * sq, q[i][2] * sq, q[i][3] * sq);
    st4(Kh + t * kLd + 4 * lane, k[i][0] * sk, k[i][1] * sk, k[i][2] * sk, k[i][3] * sk);
    if (lane == 0) {
      vb[t] = t < cl.L ? (p.beta_prob ? braw[i] : 1.f / (1.f + expf(-braw[i]))) : 0.f;
      if (rq) rq[t] = sq;
      if (rk) rk[t] = sk;
    }
  }
}

// Gamma [64][kLd]: the in-chunk cumulative sums of the activated gate (a = 0 on
// rows >= L).  kNT threads: thread = (channel, group of 64 / (kNT / 128)
// consecutive tokens); each group then adds the totals of the groups before it.
// The gate's derivatives da/dz and da/dA_log go to dz_out, da_out ([64][128],
// zero on rows >= L).  Ends with a barrier.
template <int kNT>
__device__ void gate_cumsum(const BwdParams& p, const ChunkLoc& cl, int h, float* Gm, float* dz_out,
                            float* da_out) {
  constexpr int kG = kNT / kD, kN = kC / kG;
  const int c = threadIdx.x & (kD - 1), grp = threadIdx.x >> 7;
  const float amul = gate_mul(p, h);
  const float dtb = (p.gate_mode != kGateLogspace && p.dt_bias) ? p.dt_bias[h * kD + c] : 0.f;
  float z[kN];
  const int64_t e0 = (cl.t0 * p.H + h) * kD + c, ld = p.H * kD;
  if (p.g32) {  // every load first (rows past the chunk re-read its last row)
#pragma unroll
    for (int i = 0; i < kN; ++i) z[i] = p.g32[e0 + min(kN * grp + i, cl.L - 1) * ld];
  } else {
#pragma unroll
    for (int i = 0; i < kN; ++i) z[i] = bf16_to_f(p.g[e0 + min(kN * grp + i, cl.L - 1) * ld]);
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kN; ++i) {
    const int t = kN * grp + i;
    float d1 = 0.f, d2 = 0.f;
    if (t < cl.L) acc += gate_a(p.gate_mode, z[i] + dtb, amul, p.lower_bound, d1, d2);
    Gm[t * kLd + c] = acc;
    dz_out[t * kD + c] = t < cl.L ? d1 : 0.f;
    da_out[t * kD + c] = t < cl.L ? d2 : 0.f;
  }
  __syncthreads();
  float base = 0.f;
  for (int g = 0; g < grp; ++g) base += Gm[(kN * g + kN - 1) * kLd + c];
  __syncthreads();
  if (grp) {
#pragma unroll 8
    for (int i = 0; i < kN; ++i) Gm[(kN * grp + i) * kLd + c] += base;
  }
  __syncthreads();
}

// ---- fp32 block GEMM (256 threads) ----
// Operand view: element (r, c) = p[r * ld + c] (fp32, or bf16 if b16); rows
// r >= rows read as zero.  Row starts and ld are multiples of 4 elements.
struct Opd {
  const void* p;
  int64_t ld;
  int rows, b16;
};
__device__ __forceinline__ Opd opd(const void* p, int64_t ld, int rows, int b16 = 0) {
  Opd o;
  o.p = p;
  o.ld = ld;
  o.rows = rows;
  o.b16 = b16;
  return o;
}
// elements (r, c .. c + 3), c a multiple of 4
__device__ __forceinline__ float4 opd4(const Opd& o, int r, int c) {
  if (r >= o.rows) return make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t i = (int64_t)r * o.ld + c;
  if (o.b16) {
    const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(o.p) + i);
    const float2 a = unpack_bf16(u.x), b = unpack_bf16(u.y);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return ld4(static_cast<const float*>(o.p) + i);
}

// acc[4][BN / 16] += A (64 x kd) B (kd x BN), with A(m, k) = kAT ? a(k, m) : a(m, k)
// and B(k, n) = kBT ? b(n, k) : b(k, n); kd a multiple of 16.  Thread (ty =
// lt / 16, tx = lt % 16) owns rows 4 ty + i and columns 4 tx + j (j < 4) and
// 64 + 4 tx + j - 4 (j >= 4, BN = 128).  Staged through `stage` in 16-deep
// slices read as 4-element vectors (the next slice in registers while this one
// is multiplied); begins and ends with a barrier.  256 threads of the CTA
// (local index lt) take part; every thread of the CTA must call it (it holds
// the CTA's barriers), with active = false for the others.
template <int BN, bool kAT, bool kBT>
__device__ void gemm64(float (&acc)[4][BN / 16], const Opd& a, const Opd& b, int kd, float* stage,
                       int lt, bool active) {
  constexpr int kBs = BN + 4;
  constexpr int kNB = BN / 64;   // B vectors per thread and slice
  float* As = stage;             // [16][kLs]: As[k][m]
  float* Bs = stage + 16 * kLs;  // [16][kBs]: Bs[k][n]
  const int ty = lt >> 4, tx = lt & 15;
  float4 ra, rb[kNB];
  auto fetch = [&](int k0) {  // the slice's operands into registers, one vector each
    ra = kAT ? opd4(a, k0 + (lt >> 4), 4 * (lt & 15)) : opd4(a, lt >> 2, k0 + 4 * (lt & 3));
#pragma unroll
    for (int i = 0; i < kNB; ++i) {
      const int e = lt + 256 * i;
      rb[i] = kBT ? opd4(b, e >> 2, k0 + 4 * (e & 3)) : opd4(b, k0 + e / (BN / 4), 4 * (e % (BN / 4)));
    }
  };
  f2_t c2[4][BN / 32];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < BN / 32; ++j) c2[i][j] = pk2(acc[i][2 * j], acc[i][2 * j + 1]);
  __syncthreads();  // operands written to shared memory before the call are complete
  if (active) fetch(0);
  for (int k0 = 0; k0 < kd; k0 += 16) {
    __syncthreads();  // the previous slice is consumed
    if (!active) {
      __syncthreads();
      continue;
    }
    if (kAT) {
      st4(As + (lt >> 4) * kLs + 4 * (lt & 15), ra.x, ra.y, ra.z, ra.w);
    } else {
      const int m = lt >> 2, k = 4 * (lt & 3);
      As[k * kLs + m] = ra.x;
      As[(k + 1) * kLs + m] = ra.y;
      As[(k + 2) * kLs + m] = ra.z;
      As[(k + 3) * kLs + m] = ra.w;
    }
#pragma unroll
    for (int i = 0; i < kNB; ++i) {
      const int e = lt + 256 * i;
      if (kBT) {
        const int n = e >> 2, k = 4 * (e & 3);
        Bs[k * kBs + n] = rb[i].x;
        Bs[(k + 1) * kBs + n] = rb[i].y;
        Bs[(k + 2) * kBs + n] = rb[i].z;
        Bs[(k + 3) * kBs + n] = rb[i].w;
      } else {
        st4(Bs + (e / (BN / 4)) * kBs + 4 * (e % (BN / 4)), rb[i].x, rb[i].y, rb[i].z, rb[i].w);
      }
    }
    __syncthreads();
    if (k0 + 16 < kd) fetch(k0 + 16);  // in flight during this slice's products
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 av = ld4(As + kk * kLs + 4 * ty);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      f2_t br[BN / 32];
      const ulonglong2 b0 = ld2x2(Bs + kk * kBs + 4 * tx);
      br[0] = b0.x;
      br[1] = b0.y;
      if constexpr (BN == 128) {
        const ulonglong2 b1 = ld2x2(Bs + kk * kBs + 64 + 4 * tx);
        br[2] = b1.x;
        br[3] = b1.y;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const f2_t a2 = pk2(ar[i], ar[i]);
#pragma unroll
        for (int j = 0; j < BN / 32; ++j) c2[i][j] = fma2(a2, br[j], c2[i][j]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < BN / 32; ++j) {
      const float2 v = up2(c2[i][j]);
      acc[i][2 * j] = v.x;
      acc[i][2 * j + 1] = v.y;
    }
  __syncthreads();
}

template <int N>
__device__ __forceinline__ void zero_acc(float (&acc)[4][N]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < N; ++j) acc[i][j] = 0.f;
}

// ==== 1. prep ====
constexpr int kPT = 512;  // threads of the prep and chunk-gradient kernels
constexpr int kPrepFloats = 3 * kC * kLd + 3 * kC * kLs + 80 * kLd + 2 * kStage + 3 * kC;

__global__ void __launch_bounds__(kPT, 1) kda_bwd_prep_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Kh = sm;
  float* Qh = Kh + kC * kLd;
  float* Gm = Qh + kC * kLd;
  float* Gs = Gm + kC * kLd;  // G, then T
  float* Ps = Gs + kC * kLs;
  float* Mi = Ps + kC * kLs;
  float* X = Mi + kC * kLs;   // [80][kLd]: Lk, Lq, R; the inverse's block sums; then Kg
  float* stage = X + 80 * kLd;  // two GEMM staging areas
  float* vb = stage + 2 * kStage;
  const int tid = threadIdx.x;
  const int64_t item = blockIdx.x, slot = item / p.H;
  const int h = (int)(item - slot * p.H);
  ChunkLoc cl;
  if (!locate(p, slot, cl)) return;
  float* it = p.ws + item * (int64_t)kItemFloats;

  load_rows<kPT>(p, cl, h, Kh, Qh, vb, vb + kC, vb + 2 * kC);
  __syncthreads();
  gate_cumsum<kPT>(p, cl, h, Gm, it + kItemDz, it + kItemDa);
  // normalised q, k, Gamma, beta and the norm factors, for the chunk-gradient kernel
  for (int e = tid; e < kC * 32; e += kPT) {
    const int t = e >> 5, c = 4 * (e & 31);
    *reinterpret_cast<float4*>(it + kItemQh + t * kD + c) = ld4(Qh + t * kLd + c);
    *reinterpret_cast<float4*>(it + kItemKn + t * kD + c) = ld4(Kh + t * kLd + c);
    *reinterpret_cast<float4*>(it + kItemGm + t * kD + c) = ld4(Gm + t * kLd + c);
  }
  if (tid < 3 * kC) it[kItemVec + tid] = vb[tid];

  // G and P inside the 16-token diagonal blocks, pair by pair: one thread per pair
  for (int e = tid; e < 4 * 136; e += kPT) {
    const int blk = e / 136, r = e - blk * 136;
    int ii = 0;
    while ((ii + 1) * (ii + 2) / 2 <= r) ++ii;
    const int jj = r - ii * (ii + 1) / 2;
    const int i = 16 * blk + ii, j = 16 * blk + jj;
    float sg = 0.f, sp = 0.f;
#pragma unroll 4
    for (int c = 0; c < kD; c += 4) {
      const float4 gi = ld4(Gm + i * kLd + c), gj = ld4(Gm + j * kLd + c);
      const float4 ki = ld4(Kh + i * kLd + c), kj = ld4(Kh + j * kLd + c), qi = ld4(Qh + i * kLd + c);
      const float f0 = dexp(gi.x - gj.x) * kj.x, f1 = dexp(gi.y - gj.y) * kj.y;
      const float f2 = dexp(gi.z - gj.z) * kj.z, f3 = dexp(gi.w - gj.w) * kj.w;
      sg += ki.x * f0 + ki.y * f1 + ki.z * f2 + ki.w * f3;
      sp += qi.x * f0 + qi.y * f1 + qi.z * f2 + qi.w * f3;
    }
    Gs[i * kLs + j] = j < i ? sg : 0.f;
    Ps[i * kLs + j] = sp;
  }
  for (int e = tid; e < kC * kC; e += kPT) {  // upper triangles
    const int i = e >> 6, j = e & 63;
    if (j > i) {
      Gs[i * kLs + j] = 0.f;
      Ps[i * kLs + j] = 0.f;
    }
  }
  // the blocks left of the diagonal, split at the first row r of the block
#pragma unroll 1
  for (int I = 1; I < 4; ++I) {
    const int r = 16 * I;
    float* Lk = X;
    float* Lq = X + 16 * kLd;
    float* R = X + 32 * kLd;
    __syncthreads();
    for (int e = tid; e < (32 + r) * 32; e += kPT) {
      const int row = e >> 5, c = 4 * (e & 31);
      const float4 gr = ld4(Gm + r * kLd + c);
      if (row < 32) {  // Lk / Lq rows of block I
        const int ii = row & 15, i = r + ii;
        const float4 gi = ld4(Gm + i * kLd + c);
        const float l0 = dexp(gi.x - gr.x), l1 = dexp(gi.y - gr.y), l2 = dexp(gi.z - gr.z), l3 = dexp(gi.w - gr.w);
        const float4 x = ld4((row < 16 ? Kh : Qh) + i * kLd + c);
        st4((row < 16 ? Lk : Lq) + ii * kLd + c, x.x * l0, x.y * l1, x.z * l2, x.w * l3);
      } else {
        const int j = row - 32;
        const float4 gj = ld4(Gm + j * kLd + c);
        const float4 x = ld4(Kh + j * kLd + c);
        st4(R + j * kLd + c, x.x * dexp(gr.x - gj.x), x.y * dexp(gr.y - gj.y), x.z * dexp(gr.z - gj.z),
            x.w * dexp(gr.w - gj.w));
      }
    }
    __syncthreads();
    for (int e = tid; e < 16 * r; e += kPT) {
      const int ii = e / r, j = e - ii * r;
      float sg = 0.f, sp = 0.f;
#pragma unroll 4
      for (int c = 0; c < kD; c += 4) {
        const float4 lk = ld4(Lk + ii * kLd + c), lq = ld4(Lq + ii * kLd + c), rr = ld4(R + j * kLd + c);
        sg += lk.x * rr.x + lk.y * rr.y + lk.z * rr.z + lk.w * rr.w;
        sp += lq.x * rr.x + lq.y * rr.y + lq.z * rr.z + lq.w * rr.w;
      }
      Gs[(r + ii) * kLs + j] = sg;
      Ps[(r + ii) * kLs + j] = sp;
    }
  }
  __syncthreads();
  // Minv = (I + A)^-1, A = Diag(beta) G strictly lower, by 16 x 16 blocks: the
  // diagonal blocks' inverses by forward substitution (one thread per column, in
  // registers), then block row I left of the diagonal, nearest blocks first:
  // Minv_IJ = -Minv_II sum_{J <= K < I} A_IK Minv_KJ.
  if (tid < kC) {
    const int b = tid >> 4, j = tid & 15, o = 16 * b;
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < i; ++m) acc = fmaf(Gs[(o + i) * kLs + o + m], x[m], acc);
      x[i] = (i == j ? 1.f : 0.f) - vb[o + i] * acc;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) Mi[(o + i) * kLs + o + j] = x[i];
  } else {
    for (int e = tid - kC; e < kC * kC; e += kPT - kC) {  // above the diagonal blocks
      const int i = e >> 6, j = e & 63;
      if ((j >> 4) > (i >> 4)) Mi[i * kLs + j] = 0.f;
    }
  }
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {  // block distance I - J
    float* Tm = X;               // [pairs][16][16]: sum_K A_IK Minv_KJ
    const int pairs = 4 - d;
    __syncthreads();
    for (int e = tid; e < pairs * 256; e += kPT) {
      const int J = e >> 8, I = J + d, r = (e >> 4) & 15, c = e & 15;
      float acc = 0.f;
      for (int col = 16 * J; col < 16 * I; ++col) acc = fmaf(Gs[(16 * I + r) * kLs + col], Mi[col * kLs + 16 * J + c], acc);
      Tm[e] = vb[16 * I + r] * acc;
    }
    __syncthreads();
    for (int e = tid; e < pairs * 256; e += kPT) {
      const int J = e >> 8, I = J + d, r = (e >> 4) & 15, c = e & 15;
      float acc = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) acc = fmaf(Mi[(16 * I + r) * kLs + 16 * I + m], Tm[(J << 8) + m * 16 + c], acc);
      Mi[(16 * I + r) * kLs + 16 * J + c] = -acc;
    }
  }
  __syncthreads();
  // write G, P, Minv, gC, Qg, Khat, Kg; T = Minv Diag(beta) over G; Kg into X
  for (int e = tid; e < kC * kC; e += kPT) {
    const int i = e >> 6, j = e & 63;
    it[kItemG + e] = Gs[i * kLs + j];
    it[kItemP + e] = Ps[i * kLs + j];
    it[kItemMi + e] = Mi[i * kLs + j];
  }
  __syncthreads();
  for (int e = tid; e < kC * kC; e += kPT) {
    const int i = e >> 6, j = e & 63;
    Gs[i * kLs + j] = Mi[i * kLs + j] * vb[j];
  }
  for (int e = tid; e < kC * 32; e += kPT) {
    const int t = e >> 5, c = 4 * (e & 31);
    const float4 gt = ld4(Gm + t * kLd + c), gl = ld4(Gm + (kC - 1) * kLd + c);
    const float4 kx = ld4(Kh + t * kLd + c), qx = ld4(Qh + t * kLd + c);
    const float e0 = dexp(gt.x), e1 = dexp(gt.y), e2 = dexp(gt.z), e3 = dexp(gt.w);
    st4(it + kItemQg + t * kD + c, qx.x * e0, qx.y * e1, qx.z * e2, qx.w * e3);
    st4(it + kItemKg + t * kD + c, kx.x * e0, kx.y * e1, kx.z * e2, kx.w * e3);
    st4(X + t * kLd + c, kx.x * e0, kx.y * e1, kx.z * e2, kx.w * e3);
    st4(it + kItemKh + t * kD + c, kx.x * dexp(gl.x - gt.x), kx.y * dexp(gl.y - gt.y), kx.z * dexp(gl.z - gt.z),
        kx.w * dexp(gl.w - gt.w));
  }
  if (tid < kD) it[kItemGC + tid] = dexp(Gm[(kC - 1) * kLd + tid]);
  __syncthreads();  // Qh no longer read: V (fp32, rows >= L zero) takes its place
  {
    const int lane = tid & 31, warp = tid >> 5;
    float v4[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      load4(p.v + ((cl.t0 + min(warp + 16 * i, cl.L - 1)) * p.H + h) * kD + 4 * lane, v4[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = warp + 16 * i;
      const float z = t < cl.L ? 1.f : 0.f;
      st4(Qh + t * kLd + 4 * lane, z * v4[i][0], z * v4[i][1], z * v4[i][2], z * v4[i][3]);
    }
  }
  // W = T Kg (threads 0-255) and U = T V (threads 256-511) side by side
  {
    const int half = tid >> 8, lt = tid & 255, ty = lt >> 4, tx = lt & 15;
    const Opd B = opd(half ? Qh : X, kLd, kC);
    float acc[4][8];
    zero_acc(acc);
    gemm64<128, false, false>(acc, opd(Gs, kLs, kC), B, kC, stage + half * kStage, lt, true);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float* dst = it + (half ? kItemU : kItemW) + (4 * ty + i) * kD;
      st4(dst + 4 * tx, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      st4(dst + 64 + 4 * tx, acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
  }
}

// ---- asynchronous 16-byte copies (global -> shared), per-thread groups ----
__device__ __forceinline__ void cp16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// rows x 128 fp32 (contiguous in the item) into a [rows][kLd] shared array
__device__ __forceinline__ void cp_rows128(float* dst, const float* src, int rows, int tid, int nthr) {
  for (int e = tid; e < rows * 32; e += nthr) cp16(dst + (e >> 5) * kLd + 4 * (e & 31), src + 4 * e);
}

// Channel quad k (0..15) of half h of a 128-channel row: 16-channel groups
// alternate between the halves, so that eight lanes reading rows r .. r + 3 of
// a [..][kLd] array hit eight different bank quads.
__device__ __forceinline__ int cq(int k, int h) { return 32 * (k >> 2) + 16 * h + 4 * (k & 3); }

// Channels of a product-2 thread: quads c1 = 4 chp(co) and c2 = 64 + c1, chp
// placing the two co of a quarter-warp four quads apart (with the four token
// rows of the quarter, eight different bank quads).
__device__ __forceinline__ int chp(int co) { return ((co >> 1) & 3) + 4 * (co & 1) + 8 * (co >> 3); }

constexpr int kSt = 512;                  // threads of the state passes
constexpr int kSv = 32;                   // value rows per CTA
constexpr int kSBlocks = kD / kSv;        // CTAs per (sequence, head)
constexpr int kSu = kSv + 4;              // row stride of [64][kSv] shared arrays
constexpr int kFwdFloats = 2 * kC * kLd + kC * kSv + kSv * kLd + kC * kSu + kD;
constexpr int kRevFloats = 3 * kC * kLd + kC * kLs + kSv * kLd + 2 * kC * kSu + kC * kSv / 2 + kD;

// ==== 2. forward state pass ====
// CTA = (sequence, head, 32 value rows v0 ..), 512 threads; S of the CTA's rows
// in registers (product-2 ownership) and shared memory.  Per chunk, W and the
// CTA's U columns arrive (cp.async) while the previous chunk's product 2 runs,
// Khat and gC while product 1 runs.  Both products are bound by their
// shared-memory reads, so each warp covers a block of outputs as square as the
// register budget allows.  Product 1 (Unew = U - W S^T, 64 x 32 over 128
// channels): thread = (4 tokens, 4 value rows, channel quads 4 k + quarter),
// warp = 2 token quads x 4 value quads x 4 quarters, quarters added by
// shuffles.  Product 2 (S = S Diag(gC) + Unew^T Khat, 32 x 128 over 64
// tokens): thread = (4 value rows, channel quads c1 and c1 + 64, tokens
// t = 4 i + quarter), warp = 2 value quads x 4 channel groups x 4 quarters,
// quarters added by shuffles; every quarter keeps the full result.
__global__ void __launch_bounds__(kSt, 1) kda_bwd_fwd_state_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Wb = sm;                 // W [64][kLd]
  float* Kb = Wb + kC * kLd;      // Khat [64][kLd]
  float* Ub = Kb + kC * kLd;      // U columns [64][kSv]
  float* Ss = Ub + kC * kSv;      // S [kSv][kLd]
  float* Un = Ss + kSv * kLd;     // Unew [64][kSu]
  float* gc = Un + kC * kSu;      // gC [128]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x / kSBlocks;
  const int v0 = kSv * (int)(blockIdx.x - unit * kSBlocks);
  const int64_t n = unit / p.H;
  const int h = (int)(unit - n * p.H);
  const int tq = lane & 3, co = 4 * (warp & 3) + ((lane >> 2) & 3), vq = 2 * (warp >> 2) + (lane >> 4);  // product 2
  const int c1 = 4 * chp(co), c2 = c1 + 64;
  const int cq = lane & 3, pvq = 4 * (warp & 1) + ((lane >> 2) & 3), ptq = 2 * (warp >> 1) + (lane >> 4);  // product 1
  int64_t first, count;
  seq_chunks(p, n, first, count);
  auto item = [&](int64_t ci) { return p.ws + ((first + ci) * p.H + h) * (int64_t)kItemFloats; };
  auto issue_w = [&](int64_t ci) {  // W and U columns of chunk ci
    if (ci < count) {
      const float* it = item(ci);
      cp_rows128(Wb, it + kItemW, kC, tid, kSt);
      for (int e = tid; e < kC * kSv / 4; e += kSt)
        cp16(Ub + 4 * e, it + kItemU + (e / (kSv / 4)) * kD + v0 + 4 * (e % (kSv / 4)));
    }
    cp_commit();
  };
  auto issue_k = [&](int64_t ci) {  // Khat and gC of chunk ci
    if (ci < count) {
      const float* it = item(ci);
      cp_rows128(Kb, it + kItemKh, kC, tid, kSt);
      if (tid < kD / 4) cp16(gc + 4 * tid, it + kItemGC + 4 * tid);
    }
    cp_commit();
  };
  issue_w(0);
  issue_k(0);
  float s[4][8];
  {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float x = 0.f;
        if (p.init) {
          const int64_t e = base + (int64_t)i * kD + (j < 4 ? c1 + j : c2 + j - 4);
          x = p.init_bf16 ? bf16_to_f(static_cast<const uint16_t*>(p.init)[e])
                          : static_cast<const float*>(p.init)[e];
        }
        s[i][j] = x;
      }
  }
  if (tq == 0)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(Ss + (4 * vq + i) * kLd + c1, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(Ss + (4 * vq + i) * kLd + c2, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  for (int64_t ci = 0; ci < count; ++ci) {
    float* it = item(ci);
    cp_wait<1>();     // W, U of this chunk
    __syncthreads();  // ... for every thread; Ss holds S before this chunk
    if (tq == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = it + kItemS0 + (v0 + 4 * vq + i) * kD + c1;
        st4(d, s[i][0], s[i][1], s[i][2], s[i][3]);
        st4(d + 64, s[i][4], s[i][5], s[i][6], s[i][7]);
      }
    {
      f2_t a2[4][4];  // [token i][value row j]
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a2[i][j] = 0ull;
#pragma unroll 2
      for (int ks = 0; ks < 8; ++ks) {
        const int c = 4 * (4 * ks + cq);  // quarters interleaved by quad: distinct bank groups
        ulonglong2 w[4], sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = ld2x2(Wb + (4 * ptq + i) * kLd + c);
#pragma unroll
        for (int j = 0; j < 4; ++j) sv[j] = ld2x2(Ss + (4 * pvq + j) * kLd + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) a2[i][j] = fma2(w[i].y, sv[j].y, fma2(w[i].x, sv[j].x, a2[i][j]));
      }
      float r[4] = {0.f, 0.f, 0.f, 0.f};  // the sums of token row 4 ptq + cq
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 v = up2(a2[i][j]);
          float x = v.x + v.y;
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          if (cq == i) r[j] = x;
        }
      const int t = 4 * ptq + cq;
      const float4 uu = ld4(Ub + t * kSv + 4 * pvq);
      const float n0 = uu.x - r[0], n1 = uu.y - r[1], n2 = uu.z - r[2], n3 = uu.w - r[3];
      st4(it + kItemU + t * kD + v0 + 4 * pvq, n0, n1, n2, n3);
      st4(Un + t * kSu + 4 * pvq, n0, n1, n2, n3);
    }
    __syncthreads();  // Unew complete; Wb, Ub, Ss free
    issue_w(ci + 1);
    cp_wait<1>();     // Khat, gC of this chunk
    __syncthreads();
    {
      float acc[4][8];
      {
        f2_t a2[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) a2[a][j] = 0ull;
#pragma unroll 8
        for (int i = 0; i < 16; ++i) {
          const int t = 4 * i + tq;
          const float4 u = ld4(Un + t * kSu + 4 * vq);
          const ulonglong2 k0 = ld2x2(Kb + t * kLd + c1), k1 = ld2x2(Kb + t * kLd + c2);
          const float ur[4] = {u.x, u.y, u.z, u.w};
          const f2_t kr[4] = {k0.x, k0.y, k1.x, k1.y};
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const f2_t uu = pk2(ur[a], ur[a]);
#pragma unroll
            for (int j = 0; j < 4; ++j) a2[a][j] = fma2(uu, kr[j], a2[a][j]);
          }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 v = up2(a2[a][j]);
            acc[a][2 * j] = v.x;
            acc[a][2 * j + 1] = v.y;
          }
      }
      const float4 g0 = ld4(gc + c1), g1 = ld4(gc + c2);
      const float gr[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = acc[a][j];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          s[a][j] = fmaf(s[a][j], gr[j], x);
        }
      if (tq == 0)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          st4(Ss + (4 * vq + a) * kLd + c1, s[a][0], s[a][1], s[a][2], s[a][3]);
          st4(Ss + (4 * vq + a) * kLd + c2, s[a][4], s[a][5], s[a][6], s[a][7]);
        }
    }
    __syncthreads();  // Kb, gc, Un free
    issue_k(ci + 1);
  }
  cp_wait<0>();
}

// ==== 3. reverse state pass ====
// Same grid, threads and warp shapes as the forward pass, chunks last to first.
// Per chunk, Khat, P, the CTA's dout columns and gC arrive while the previous
// chunk's product B runs, Qg and W while product A runs.  Product A (dU =
// scale P^T dO + Khat dS^T, 64 x 32): thread = (4 tokens, 4 value rows, quarter
// of the channel quads and of the tokens j).  Product B (dS = dS Diag(gC) +
// scale dO^T Qg - dU^T W, 32 x 128 over 64 tokens) as the forward pass's
// product 2.
__global__ void __launch_bounds__(kSt, 1) kda_bwd_rev_state_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Kb = sm;                 // Khat [64][kLd]
  float* Qb = Kb + kC * kLd;      // Qg
  float* Wb = Qb + kC * kLd;      // W
  float* Pb = Wb + kC * kLd;      // P [64][kLs]
  float* Ds = Pb + kC * kLs;      // dS [kSv][kLd]
  float* Os = Ds + kSv * kLd;     // scale dO [64][kSu]
  float* Us = Os + kC * kSu;      // dU [64][kSu]
  uint16_t* Ob = reinterpret_cast<uint16_t*>(Us + kC * kSu);  // dO bf16 [64][kSv]
  float* gc = Us + kC * kSu + kC * kSv / 2;                      // gC [128]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x / kSBlocks;
  const int v0 = kSv * (int)(blockIdx.x - unit * kSBlocks);
  const int64_t n = unit / p.H;
  const int h = (int)(unit - n * p.H);
  const int tq = lane & 3, co = 4 * (warp & 3) + ((lane >> 2) & 3), vq = 2 * (warp >> 2) + (lane >> 4);
  const int c1 = 4 * chp(co), c2 = c1 + 64;
  const int cq = lane & 3, pvq = 4 * (warp & 1) + ((lane >> 2) & 3), ptq = 2 * (warp >> 1) + (lane >> 4);
  int64_t first, count;
  seq_chunks(p, n, first, count);
  const int64_t bos = p.cu ? p.cu[n] : n * p.T, eos = p.cu ? p.cu[n + 1] : (n + 1) * p.T;
  auto item = [&](int64_t ci) { return p.ws + ((first + ci) * p.H + h) * (int64_t)kItemFloats; };
  auto chunk_len = [&](int64_t ci) { return (int)min((int64_t)kC, eos - bos - ci * kC); };
  auto issue_a = [&](int64_t ci) {  // Khat, P, dout columns, gC of chunk ci
    if (ci >= 0) {
      const float* it = item(ci);
      cp_rows128(Kb, it + kItemKh, kC, tid, kSt);
      for (int e = tid; e < kC * 16; e += kSt) cp16(Pb + (e >> 4) * kLs + 4 * (e & 15), it + kItemP + 4 * e);
      const int L = chunk_len(ci);
      for (int e = tid; e < L * (kSv / 8); e += kSt) {
        const int t = e / (kSv / 8), q = e % (kSv / 8);
        cp16(Ob + t * kSv + 8 * q, p.dout + ((bos + ci * kC + t) * p.H + h) * kD + v0 + 8 * q);
      }
      if (tid < kD / 4) cp16(gc + 4 * tid, it + kItemGC + 4 * tid);
    }
    cp_commit();
  };
  auto issue_b = [&](int64_t ci) {  // Qg and W of chunk ci
    if (ci >= 0) {
      const float* it = item(ci);
      cp_rows128(Qb, it + kItemQg, kC, tid, kSt);
      cp_rows128(Wb, it + kItemW, kC, tid, kSt);
    }
    cp_commit();
  };
  issue_a(count - 1);
  issue_b(count - 1);
  float s[4][8];
  {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j)
        s[i][j] = p.dfinal ? p.dfinal[base + (int64_t)i * kD + (j < 4 ? c1 + j : c2 + j - 4)] : 0.f;
  }
  if (tq == 0)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(Ds + (4 * vq + i) * kLd + c1, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(Ds + (4 * vq + i) * kLd + c2, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  for (int64_t ci = count - 1; ci >= 0; --ci) {
    float* it = item(ci);
    const int L = chunk_len(ci);
    cp_wait<1>();     // Khat, P, dout, gC of this chunk
    __syncthreads();  // ... for every thread; Ds holds dS_C
    for (int e = tid; e < kC * kSv; e += kSt) {
      const int t = e / kSv, v = e % kSv;
      Os[t * kSu + v] = t < L ? p.scale * bf16_to_f(Ob[e]) : 0.f;
    }
    if (tq == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = it + kItemDS + (v0 + 4 * vq + i) * kD + c1;
        st4(d, s[i][0], s[i][1], s[i][2], s[i][3]);
        st4(d + 64, s[i][4], s[i][5], s[i][6], s[i][7]);
      }
    __syncthreads();
    {
      f2_t a2[4][4];  // [token i][value row j]: Khat dS^T over this quarter's channel quads
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a2[i][j] = 0ull;
#pragma unroll 2
      for (int ks = 0; ks < 8; ++ks) {
        const int c = 4 * (4 * ks + cq);
        ulonglong2 kk[4], dd[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) kk[i] = ld2x2(Kb + (4 * ptq + i) * kLd + c);
#pragma unroll
        for (int j = 0; j < 4; ++j) dd[j] = ld2x2(Ds + (4 * pvq + j) * kLd + c);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) a2[i][j] = fma2(kk[i].y, dd[j].y, fma2(kk[i].x, dd[j].x, a2[i][j]));
      }
      float acc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 v = up2(a2[i][j]);
          acc[i][j] = v.x + v.y;
        }
#pragma unroll 4
      for (int j = cq; j < kC; j += 4) {  // scale P^T dO over this quarter's tokens j
        const float4 pj = ld4(Pb + j * kLs + 4 * ptq);
        const float4 o = ld4(Os + j * kSu + 4 * pvq);
        const float pr[4] = {pj.x, pj.y, pj.z, pj.w}, orr[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(pr[i], orr[jj], acc[i][jj]);
      }
      float r[4] = {0.f, 0.f, 0.f, 0.f};  // the sums of token row 4 ptq + cq
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float x = acc[i][j];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          if (cq == i) r[j] = x;
        }
      const int t = 4 * ptq + cq;
      st4(it + kItemDU + t * kD + v0 + 4 * pvq, r[0], r[1], r[2], r[3]);
      st4(Us + t * kSu + 4 * pvq, r[0], r[1], r[2], r[3]);
    }
    __syncthreads();  // dU complete; Kb, Pb, Ob, Ds free
    const float4 g0 = ld4(gc + c1), g1 = ld4(gc + c2);
    __syncthreads();  // gc read by every thread before it is replaced
    issue_a(ci - 1);
    cp_wait<1>();     // Qg, W of this chunk
    __syncthreads();
    {
      float acc[4][8];
      {
        f2_t a2[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) a2[a][j] = 0ull;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          const int t = 4 * i + tq;
          const float4 o = ld4(Os + t * kSu + 4 * vq), u = ld4(Us + t * kSu + 4 * vq);
          const ulonglong2 q0 = ld2x2(Qb + t * kLd + c1), q1 = ld2x2(Qb + t * kLd + c2);
          const ulonglong2 w0 = ld2x2(Wb + t * kLd + c1), w1 = ld2x2(Wb + t * kLd + c2);
          const float orr[4] = {o.x, o.y, o.z, o.w}, ur[4] = {u.x, u.y, u.z, u.w};
          const f2_t qr[4] = {q0.x, q0.y, q1.x, q1.y}, wr[4] = {w0.x, w0.y, w1.x, w1.y};
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            const f2_t oo = pk2(orr[a], orr[a]), uu = pk2(-ur[a], -ur[a]);
#pragma unroll
            for (int j = 0; j < 4; ++j) a2[a][j] = fma2(oo, qr[j], fma2(uu, wr[j], a2[a][j]));
          }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 v = up2(a2[a][j]);
            acc[a][2 * j] = v.x;
            acc[a][2 * j + 1] = v.y;
          }
      }
      const float gr[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = acc[a][j];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          s[a][j] = fmaf(s[a][j], gr[j], x);
        }
      if (tq == 0)
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          st4(Ds + (4 * vq + a) * kLd + c1, s[a][0], s[a][1], s[a][2], s[a][3]);
          st4(Ds + (4 * vq + a) * kLd + c2, s[a][4], s[a][5], s[a][6], s[a][7]);
        }
    }
    __syncthreads();  // Qb, Wb, Os, Us free
    issue_b(ci - 1);
  }
  cp_wait<0>();
  if (p.dinit && tq == 0) {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(p.dinit + base + (int64_t)i * kD + c1, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(p.dinit + base + (int64_t)i * kD + c2, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  }
}

// ==== 4. gradient products ====
__global__ void __launch_bounds__(256, 3) kda_bwd_prod_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* dWs = sm;  // [64][kLd]
  float* stage = dWs + kC * kLd;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t item = blockIdx.x, slot = item / p.H;
  const int h = (int)(item - slot * p.H);
  ChunkLoc cl;
  if (!locate(p, slot, cl)) return;
  float* it = p.ws + item * (int64_t)kItemFloats;
  const int64_t rbase = (cl.t0 * p.H + h) * kD;  // element (t, x) of a token tensor at rbase + t H 128 + x
  const Opd dO = opd(p.dout + rbase, p.H * kD, cl.L, 1);
  const Opd Vv = opd(p.v + rbase, p.H * kD, cl.L, 1);
  const Opd S0 = opd(it + kItemS0, kD, kD), dS = opd(it + kItemDS, kD, kD);
  const Opd Un = opd(it + kItemU, kD, kC), dU = opd(it + kItemDU, kD, kC);
  const Opd Mi = opd(it + kItemMi, kC, kC), Kg = opd(it + kItemKg, kD, kC);
  auto store128 = [&](float* dst, const float (&acc)[4][8], float mul) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float* d = dst + (4 * ty + i) * kD;
      st4(d + 4 * tx, mul * acc[i][0], mul * acc[i][1], mul * acc[i][2], mul * acc[i][3]);
      st4(d + 64 + 4 * tx, mul * acc[i][4], mul * acc[i][5], mul * acc[i][6], mul * acc[i][7]);
    }
  };
  float acc[4][8];
  // dQg = scale dO S (over Qg, no longer read)
  zero_acc(acc);
  gemm64<128, false, false>(acc, dO, S0, kD, stage, tid, true);
  store128(it + kItemQg, acc, p.scale);
  // dW = -dU S (shared memory)
  zero_acc(acc);
  gemm64<128, false, false>(acc, dU, S0, kD, stage, tid, true);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* d = dWs + (4 * ty + i) * kLd;
    st4(d + 4 * tx, -acc[i][0], -acc[i][1], -acc[i][2], -acc[i][3]);
    st4(d + 64 + 4 * tx, -acc[i][4], -acc[i][5], -acc[i][6], -acc[i][7]);
  }
  // dKhat = Unew dS_C
  zero_acc(acc);
  gemm64<128, false, false>(acc, Un, dS, kD, stage, tid, true);
  store128(it + kItemKh, acc, 1.f);
  // dgC = colsum(S . dS_C): two threads per channel, halves added through
  // shared memory (the staging area, free between products)
  {
    const int c = tid & (kD - 1), v0 = 64 * (tid >> 7);
    float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
    for (int v = v0; v < v0 + 64; v += 8)
#pragma unroll
      for (int u = 0; u < 8; ++u) x[u] = fmaf(it[kItemS0 + (v + u) * kD + c], it[kItemDS + (v + u) * kD + c], x[u]);
    const float y = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    if (tid >= kD) stage[c] = y;
    __syncthreads();
    if (tid < kD) it[kItemDGC + c] = y + stage[c];
  }
  // dP = scale dO Unew^T (s <= t)
  {
    float a2[4][4];
    zero_acc(a2);
    gemm64<64, false, true>(a2, dO, Un, kD, stage, tid, true);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * ty + i;
      float x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = (4 * tx + j <= t) ? p.scale * a2[i][j] : 0.f;
      st4(it + kItemP + t * kC + 4 * tx, x[0], x[1], x[2], x[3]);
    }
  }
  // dT = dU V^T + dW Kg^T (s <= t)
  {
    float a2[4][4];
    zero_acc(a2);
    gemm64<64, false, true>(a2, dU, Vv, kD, stage, tid, true);
    gemm64<64, false, true>(a2, opd(dWs, kLd, kC), Kg, kD, stage, tid, true);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * ty + i;
      float x[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) x[j] = (4 * tx + j <= t) ? a2[i][j] : 0.f;
      st4(it + kItemDT + t * kC + 4 * tx, x[0], x[1], x[2], x[3]);
    }
  }
  // beta of the rows this thread stores
  float bt[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 4 * ty + i;
    float b = 0.f;
    if (t < cl.L) {
      const float braw = bf16_to_f(p.beta[(cl.t0 + t) * p.H + h]);
      b = p.beta_prob ? braw : 1.f / (1.f + expf(-braw));
    }
    bt[i] = b;
  }
  // dv = Diag(beta) Minv^T dU
  zero_acc(acc);
  gemm64<128, true, false>(acc, Mi, dU, kC, stage, tid, true);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = 4 * ty + i;
    if (t < cl.L) {
      float* d = p.dv + rbase + (int64_t)t * p.H * kD;
      st4(d + 4 * tx, bt[i] * acc[i][0], bt[i] * acc[i][1], bt[i] * acc[i][2], bt[i] * acc[i][3]);
      st4(d + 64 + 4 * tx, bt[i] * acc[i][4], bt[i] * acc[i][5], bt[i] * acc[i][6], bt[i] * acc[i][7]);
    }
  }
  // dKg = Diag(beta) Minv^T dW (over W, no longer read)
  zero_acc(acc);
  gemm64<128, true, false>(acc, Mi, opd(dWs, kLd, kC), kC, stage, tid, true);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* d = it + kItemW + (4 * ty + i) * kD;
    st4(d + 4 * tx, bt[i] * acc[i][0], bt[i] * acc[i][1], bt[i] * acc[i][2], bt[i] * acc[i][3]);
    st4(d + 64 + 4 * tx, bt[i] * acc[i][4], bt[i] * acc[i][5], bt[i] * acc[i][6], bt[i] * acc[i][7]);
  }
}

// ==== 5. chunk gradients ====
// 512 threads: thread (hf = tid / 256, ty = (tid % 256) / 16, tx = tid % 16)
// accumulates dq_hat, dk_hat and dGamma of rows 16 m + ty (m = 0..3), channels
// cb = 64 hf + 4 tx .. cb + 3, in registers.
constexpr int kGradFloats = 3 * kC * kLd + 2 * kC * kLs + 80 * kLd + kStage + 16 * kD + 4 * kC + 4 * kC;

__device__ __forceinline__ void f4a(float4 v, float (&x)[4]) {
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}

__global__ void __launch_bounds__(kPT, 1) kda_bwd_grad_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Kh = sm;
  float* Qh = Kh + kC * kLd;
  float* Gm = Qh + kC * kLd;
  float* dGs = Gm + kC * kLd;  // dG [64][kLs]
  float* dPs = dGs + kC * kLs;  // dP
  float* X = dPs + kC * kLs;    // [80][kLd] scratch
  float* stage = X + 80 * kLd;
  float* part = stage + kStage;  // [16][128]
  float* vb = part + 16 * kD;
  float* rq = vb + kC;
  float* rk = rq + kC;
  float* dbv = rk + kC;
  float* xs = dbv + kC;          // [2 halves][2][64]: row sums of the norm terms
  const int tid = threadIdx.x, hf = tid >> 8, lt = tid & 255, ty = lt >> 4, tx = lt & 15;
  const int cb = 64 * hf + 4 * tx;
  const int64_t item = blockIdx.x, slot = item / p.H;
  const int h = (int)(item - slot * p.H);
  ChunkLoc cl;
  if (!locate(p, slot, cl)) return;
  float* it = p.ws + item * (int64_t)kItemFloats;
  // the chunk's rows as the recompute left them (normalised k, q, Gamma; beta
  // and the norm factors), dT, Minv and P (Minv where dG goes later, dT at the
  // start of the scratch area), into shared memory
  for (int e = tid; e < kC * 32; e += kPT) {
    const int t = e >> 5, c = 4 * (e & 31);
    cp16(Kh + t * kLd + c, it + kItemKn + 4 * e);
    cp16(Qh + t * kLd + c, it + kItemQh + 4 * e);
    cp16(Gm + t * kLd + c, it + kItemGm + 4 * e);
  }
  for (int e = tid; e < kC * 16; e += kPT) {
    const int i = e >> 4, c = 4 * (e & 15);
    cp16(X + i * kLs + c, it + kItemDT + 4 * e);
    cp16(dGs + i * kLs + c, it + kItemMi + 4 * e);
    cp16(dPs + i * kLs + c, it + kItemP + 4 * e);
  }
  if (tid < 3 * kC / 4) cp16(vb + 4 * tid, it + kItemVec + 4 * tid);  // vb, rq, rk contiguous
  cp_commit();

  // ---- dM = -Minv^T (dT Diag(beta)) Minv^T, dA, dG, dbeta (threads 0-255) ----
  {
    float* Mi = dGs;            // Minv [64][kLs] until dG replaces it
    float* Xa = X;              // dT
    float* Xb = X + kC * kLs;   // (Minv^T dT) Diag(beta)
    cp_wait<0>();
    __syncthreads();
    const bool act = hf == 0;
    float a2[4][4];
    zero_acc(a2);
    gemm64<64, true, false>(a2, opd(Mi, kLs, kC), opd(Xa, kLs, kC), kC, stage, lt, act);
    if (act) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (ty == tx) dbv[4 * ty + i] = a2[i][i];  // (Minv^T dT)_tt
        st4(Xb + (4 * ty + i) * kLs + 4 * tx, a2[i][0] * vb[4 * tx], a2[i][1] * vb[4 * tx + 1],
            a2[i][2] * vb[4 * tx + 2], a2[i][3] * vb[4 * tx + 3]);
      }
    }
    zero_acc(a2);
    gemm64<64, false, true>(a2, opd(Xb, kLs, kC), opd(Mi, kLs, kC), kC, stage, lt, act);
    if (act) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * ty + i;
        float gv[4];
        f4a(ld4(it + kItemG + t * kC + 4 * tx), gv);
        float d[4], gsum = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = 4 * tx + j;
          const float dA = s < t ? -a2[i][j] : 0.f;
          gsum = fmaf(dA, gv[j], gsum);
          d[j] = vb[t] * dA;
        }
        st4(dGs + t * kLs + 4 * tx, d[0], d[1], d[2], d[3]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
        if (tx == 0) dbv[t] += gsum;
      }
    }
  }
  __syncthreads();

  // The pairwise sums G and P contribute, per row t and channel c, three sums:
  //   xi = sum_{s<t} dG_ts k_s F_ts     (t the later token of a G term)
  //   xp = sum_{s<=t} dP_ts k_s F_ts    (t the later token of a P term)
  //   yj = sum_{i>t} (dG_it k_i + dP_it q_i) F_it   (t the earlier token; i = t for P)
  // giving dk += xi + yj, dq += xp and dGamma += k xi + q xp - k yj.  Registers:
  // aK = xi, aQ = xp, aG = yj until the scalings below combine them.
  float aQ[4][4], aK[4][4], aG[4][4];
#pragma unroll
  for (int m = 0; m < 4; ++m)
#pragma unroll
    for (int j = 0; j < 4; ++j) aQ[m][j] = aK[m][j] = aG[m][j] = 0.f;
  // ---- G and P inside the diagonal blocks, pair by pair ----
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int t = 16 * m + ty;
    float gt[4], kt[4], qt[4];
    f4a(ld4(Gm + t * kLd + cb), gt);
    f4a(ld4(Kh + t * kLd + cb), kt);
    f4a(ld4(Qh + t * kLd + cb), qt);
    const float dpd = dPs[t * kLs + t];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      aQ[m][j] = dpd * kt[j];
      aG[m][j] = dpd * qt[j];
    }
#pragma unroll 4
    for (int s = 16 * m; s < 16 * m + 16; ++s) {
      if (s == t) continue;
      float gs[4], ks[4];
      f4a(ld4(Gm + s * kLd + cb), gs);
      f4a(ld4(Kh + s * kLd + cb), ks);
      if (s < t) {  // t takes the role of the later token
        const float dg = dGs[t * kLs + s], dp = dPs[t * kLs + s];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float f = dexp(gt[j] - gs[j]) * ks[j];
          aK[m][j] = fmaf(dg, f, aK[m][j]);
          aQ[m][j] = fmaf(dp, f, aQ[m][j]);
        }
      } else {  // t is the earlier token
        const float dg = dGs[s * kLs + t], dp = dPs[s * kLs + t];
        float qs[4];
        f4a(ld4(Qh + s * kLd + cb), qs);
#pragma unroll
        for (int j = 0; j < 4; ++j) aG[m][j] = fmaf(fmaf(dg, ks[j], dp * qs[j]), dexp(gs[j] - gt[j]), aG[m][j]);
      }
    }
  }
  // ---- blocks left of the diagonal, split at the first row r of block I ----
#pragma unroll
  for (int I = 1; I < 4; ++I) {
    const int r = 16 * I;
    float* Lk = X;
    float* Lq = X + 16 * kLd;
    float* R = X + 32 * kLd;
    __syncthreads();
    for (int e = tid; e < (32 + r) * 32; e += kPT) {
      const int row = e >> 5, c = 4 * (e & 31);
      const float4 gr = ld4(Gm + r * kLd + c);
      if (row < 32) {
        const int ii = row & 15, i = r + ii;
        const float4 gi = ld4(Gm + i * kLd + c);
        const float4 x = ld4((row < 16 ? Kh : Qh) + i * kLd + c);
        st4((row < 16 ? Lk : Lq) + ii * kLd + c, x.x * dexp(gi.x - gr.x), x.y * dexp(gi.y - gr.y),
            x.z * dexp(gi.z - gr.z), x.w * dexp(gi.w - gr.w));
      } else {
        const int j = row - 32;
        const float4 gj = ld4(Gm + j * kLd + c);
        const float4 x = ld4(Kh + j * kLd + c);
        st4(R + j * kLd + c, x.x * dexp(gr.x - gj.x), x.y * dexp(gr.y - gj.y), x.z * dexp(gr.z - gj.z),
            x.w * dexp(gr.w - gj.w));
      }
    }
    __syncthreads();
    {  // rows of block I (t = r + ty): xi += l (dG R), xp += l (dP R) over s < r, l = e^{Gamma_t - Gamma_r}
      const int t = r + ty;
      float xg[4] = {0.f, 0.f, 0.f, 0.f}, xp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int s = 0; s < r; ++s) {
        const float dg = dGs[t * kLs + s], dp = dPs[t * kLs + s];
        float rr[4];
        f4a(ld4(R + s * kLd + cb), rr);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          xg[j] = fmaf(dg, rr[j], xg[j]);
          xp[j] = fmaf(dp, rr[j], xp[j]);
        }
      }
      float gtv[4], grv[4];
      f4a(ld4(Gm + t * kLd + cb), gtv);
      f4a(ld4(Gm + r * kLd + cb), grv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float l = dexp(gtv[j] - grv[j]);
        aK[I][j] = fmaf(l, xg[j], aK[I][j]);
        aQ[I][j] = fmaf(l, xp[j], aQ[I][j]);
      }
    }
#pragma unroll
    for (int m = 0; m < I; ++m) {  // rows s = 16 m + ty < r: yj += e^{Gamma_r - Gamma_s} (dG^T Lk + dP^T Lq)
      const int s = 16 * m + ty;
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int ii = 0; ii < 16; ++ii) {
        const float dg = dGs[(r + ii) * kLs + s], dp = dPs[(r + ii) * kLs + s];
        float kr[4], qr[4];
        f4a(ld4(Lk + ii * kLd + cb), kr);
        f4a(ld4(Lq + ii * kLd + cb), qr);
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = fmaf(dg, kr[j], fmaf(dp, qr[j], y[j]));
      }
      float grv[4], gsv[4];
      f4a(ld4(Gm + r * kLd + cb), grv);
      f4a(ld4(Gm + s * kLd + cb), gsv);
#pragma unroll
      for (int j = 0; j < 4; ++j) aG[m][j] = fmaf(dexp(grv[j] - gsv[j]), y[j], aG[m][j]);
    }
  }
  // ---- the scalings Qg = q e^Gamma, Kg = k e^Gamma, Khat = k e^{Gamma_C - Gamma}, and the
  // combination of the pairwise sums ----
  {
    float cs[4] = {0.f, 0.f, 0.f, 0.f};
    float4 gq[4], gk[4], gh[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {  // every load first
      const int o = (16 * m + ty) * kD + cb;
      gq[m] = ld4(it + kItemQg + o);
      gk[m] = ld4(it + kItemW + o);
      gh[m] = ld4(it + kItemKh + o);
    }
    float glv[4];
    f4a(ld4(Gm + (kC - 1) * kLd + cb), glv);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int t = 16 * m + ty;
      float dqv[4], dkv[4], dhv[4], gtv[4], qhv[4], khv[4];
      f4a(gq[m], dqv);
      f4a(gk[m], dkv);
      f4a(gh[m], dhv);
      f4a(ld4(Gm + t * kLd + cb), gtv);
      f4a(ld4(Qh + t * kLd + cb), qhv);
      f4a(ld4(Kh + t * kLd + cb), khv);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float e = dexp(gtv[j]), ec = dexp(glv[j] - gtv[j]);
        const float xi = aK[m][j], xp = aQ[m][j], yj = aG[m][j];
        aQ[m][j] = xp + dqv[j] * e;
        aK[m][j] = xi + yj + dkv[j] * e + dhv[j] * ec;
        aG[m][j] = khv[j] * (xi - yj) + qhv[j] * xp + dqv[j] * qhv[j] * e + dkv[j] * khv[j] * e -
                   dhv[j] * khv[j] * ec;
        cs[j] += dhv[j] * khv[j] * ec;
      }
    }
    st4(part + ty * kD + cb, cs[0], cs[1], cs[2], cs[3]);
  }
  __syncthreads();
  // ---- dGamma -> da by the reverse cumulative sum; row sums of the norm terms ----
  float* Dg = X;  // [64][kLd]
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int t = 16 * m + ty;
    st4(Dg + t * kLd + cb, aG[m][0], aG[m][1], aG[m][2], aG[m][3]);
    float qv[4], kv[4];
    f4a(ld4(Qh + t * kLd + cb), qv);
    f4a(ld4(Kh + t * kLd + cb), kv);
    float xq = 0.f, xk = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      xq = fmaf(qv[j], aQ[m][j], xq);
      xk = fmaf(kv[j], aK[m][j], xk);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      xq += __shfl_xor_sync(0xffffffffu, xq, o);
      xk += __shfl_xor_sync(0xffffffffu, xk, o);
    }
    if (tx == 0) {
      xs[(hf * 2) * kC + t] = xq;
      xs[(hf * 2 + 1) * kC + t] = xk;
    }
  }
  __syncthreads();
  if (tid < kD) {
    float x = it[kItemDGC + tid] * dexp(Gm[(kC - 1) * kLd + tid]);
    for (int y = 0; y < 16; ++y) x += part[y * kD + tid];
    float acc = Dg[(kC - 1) * kLd + tid] + x;
    Dg[(kC - 1) * kLd + tid] = acc;
    for (int t = kC - 2; t >= 0; --t) {
      acc += Dg[t * kLd + tid];
      Dg[t * kLd + tid] = acc;
    }
  }
  __syncthreads();
  // ---- outputs ----
  float pdt[4] = {0.f, 0.f, 0.f, 0.f}, pal = 0.f;
  float4 dzall[4], daall[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {  // every load first: the gate's derivatives from the recompute
    dzall[m] = ld4(it + kItemDz + (16 * m + ty) * kD + cb);
    daall[m] = ld4(it + kItemDa + (16 * m + ty) * kD + cb);
  }
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int t = 16 * m + ty;
    if (t >= cl.L) continue;
    const int64_t row = (cl.t0 + t) * p.H + h;
    float qv[4], kv[4], dav[4], dzv[4], dAv[4];
    f4a(ld4(Qh + t * kLd + cb), qv);
    f4a(ld4(Kh + t * kLd + cb), kv);
    f4a(ld4(Dg + t * kLd + cb), dav);
    f4a(dzall[m], dzv);
    f4a(daall[m], dAv);
    const float xq = xs[t] + xs[2 * kC + t], xk = xs[kC + t] + xs[3 * kC + t];
    float dq[4], dk[4], dz[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (p.l2norm) {
        dq[j] = rq[t] * (aQ[m][j] - qv[j] * xq);
        dk[j] = rk[t] * (aK[m][j] - kv[j] * xk);
      } else {
        dq[j] = aQ[m][j];
        dk[j] = aK[m][j];
      }
      dz[j] = dav[j] * dzv[j];
      pdt[j] += dz[j];
      pal = fmaf(dav[j], dAv[j], pal);
    }
    st4(p.dq + row * kD + cb, dq[0], dq[1], dq[2], dq[3]);
    st4(p.dk + row * kD + cb, dk[0], dk[1], dk[2], dk[3]);
    st4(p.dg + row * kD + cb, dz[0], dz[1], dz[2], dz[3]);
  }
  if (tid < cl.L) {
    float db = dbv[tid];
    if (!p.beta_prob) db *= vb[tid] * (1.f - vb[tid]);
    p.dbeta[(cl.t0 + tid) * p.H + h] = db;
  }
  // the chunk's parts of dt_bias and A_log, summed in a fixed order
  __syncthreads();
  st4(part + ty * kD + cb, pdt[0], pdt[1], pdt[2], pdt[3]);
  pal = warp_sum(pal);
  if ((tid & 31) == 0) X[tid >> 5] = pal;
  __syncthreads();
  if (tid < kD) {
    float x = 0.f;
    for (int y = 0; y < 16; ++y) x += part[y * kD + tid];
    it[kItemPart + tid] = x;
  }
  if (tid == kD) {
    float x = 0.f;
    for (int w = 0; w < kPT / 32; ++w) x += X[w];
    it[kItemPart + kD] = x;
  }
}

// ==== 6. finalize: dA_log and dt_bias, the chunks' parts in slot order ====
__global__ void __launch_bounds__(kD + 32) kda_bwd_finalize_kernel(BwdParams p) {
  const int h = blockIdx.x, tid = threadIdx.x;
  const int64_t slots = p.cu ? p.chunk_off[p.N] : p.nslots;
  if (tid > kD) return;
  float x = 0.f;
  for (int64_t s = 0; s < slots; ++s) x += p.ws[(s * p.H + h) * (int64_t)kItemFloats + kItemPart + tid];
  if (tid < kD) {
    if (p.ddt_bias) p.ddt_bias[h * kD + tid] = x;
  } else if (p.dA_log) {
    p.dA_log[h] = p.A_log ? x : 0.f;  // without A_log the gate has no such parameter
  }
}

}  // namespace

// Items (chunk slots x heads) and the launches.  ev: optional events
// (cudaEvent_t, each may be null) recorded after the forward state pass, the
// reverse state pass and the finalize launch (entries 1, 2, 3).
static void launch_bwd(const BwdParams& p, cudaStream_t s, void* const* ev) {
  auto mark = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s);
  };
  const unsigned items = (unsigned)(p.nslots * p.H);
  const unsigned units = (unsigned)(p.N * p.H * kSBlocks);
  if (items) kda_bwd_prep_kernel<<<items, kPT, kPrepFloats * 4, s>>>(p);
  kda_bwd_fwd_state_kernel<<<units, kSt, kFwdFloats * 4, s>>>(p);
  mark(1);
  kda_bwd_rev_state_kernel<<<units, kSt, kRevFloats * 4, s>>>(p);
  mark(2);
  if (items) {
    kda_bwd_prod_kernel<<<items, 256, kProdFloats * 4, s>>>(p);
    kda_bwd_grad_kernel<<<items, kPT, kGradFloats * 4, s>>>(p);
  }
  if (p.gate_mode != kGateLogspace && (p.dA_log || p.ddt_bias))
    kda_bwd_finalize_kernel<<<(unsigned)p.H, kD + 32, 0, s>>>(p);
  mark(3);
}

static cudaError_t prepare_bwd() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute((const void*)kda_bwd_prep_kernel, attr, kPrepFloats * 4);
  if (e == cudaSuccess) e = cudaFuncSetAttribute((const void*)kda_bwd_prod_kernel, attr, kProdFloats * 4);
  if (e == cudaSuccess) e = cudaFuncSetAttribute((const void*)kda_bwd_grad_kernel, attr, kGradFloats * 4);
  if (e == cudaSuccess) e = cudaFuncSetAttribute((const void*)kda_bwd_fwd_state_kernel, attr, kFwdFloats * 4);
  if (e == cudaSuccess) e = cudaFuncSetAttribute((const void*)kda_bwd_rev_state_kernel, attr, kRevFloats * 4);
  return e;
}

}  // namespace kda

// ---- host entry points ----
using namespace kda;

namespace {
std::atomic<int> g_bwd_prepared[64];
// The forward arguments as kda_fwd checks them; out is not used by the
// backward pass, so dout stands in for it.
int validate_bwd(const kda_bwd_args* a, int64_t* slots, size_t* header) {
  kda_fwd_args f = a->fwd;
  f.out = const_cast<void*>(a->dout);
  f.final_state = nullptr;
  return validate(&f, slots, header);
}
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned16(const void* p) { return p == nullptr || ((uintptr_t)p % 16) == 0; }
}  // namespace

extern "C" size_t kda_bwd_workspace_bytes(const kda_bwd_args* a) {
  if (!a) return 0;
  int64_t slots = 0;
  size_t header = 0;
  if (validate_bwd(a, &slots, &header) != KDA_OK) return 0;
  return round256(header) + (size_t)slots * (size_t)a->fwd.H * kItemFloats * sizeof(float);
}

namespace {
int bwd_device(const kda_bwd_args* a, void* workspace, size_t workspace_bytes, void* stream_ptr,
               void* const* events) {
  if (!a) return KDA_ERR_NULL_ARG;
  const kda_fwd_args& f = a->fwd;
  int64_t slots = 0;
  size_t header = 0;
  const int rc = validate_bwd(a, &slots, &header);
  if (rc != KDA_OK) return rc;
  const int64_t rows = f.B * f.T;
  if (rows > 0 && (!a->dout || !a->dq || !a->dk || !a->dv || !a->dg || !a->dbeta)) return KDA_ERR_NULL_ARG;
  if (!aligned16(a->dout) || !aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv) ||
      !aligned16(a->dg) || !aligned16(a->dfinal_state) || !aligned16(a->ddt_bias) ||
      !aligned16(a->dinitial_state) || (a->dbeta && ((uintptr_t)a->dbeta % 4)) ||
      (a->dA_log && ((uintptr_t)a->dA_log % 4)))
    return KDA_ERR_ALIGNMENT;
  if (f.N == 0 || f.H == 0) return KDA_OK;
  const size_t need = kda_bwd_workspace_bytes(a);
  if (!workspace || ((uintptr_t)workspace % 256) || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_LAUNCH;
  if (g_bwd_prepared[dev].load() == 0) {
    if (prepare_bwd() != cudaSuccess) return KDA_ERR_LAUNCH;
    g_bwd_prepared[dev].store(1);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream_ptr);
  int* status = status_slot(s);
  if (!status) return KDA_ERR_LAUNCH;
  if (events && events[0]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(events[0]), s);
  const int64_t H = f.H;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const uint32_t gate = f.flags & (KDA_GATE_SAFE | KDA_GATE_UNSAFE | KDA_GATE_LOGSPACE);
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  BwdParams p;
  p.q = static_cast<const uint16_t*>(f.q);
  p.k = static_cast<const uint16_t*>(f.k);
  p.v = static_cast<const uint16_t*>(f.v);
  p.g = static_cast<const uint16_t*>(f.g);
  p.g32 = (f.flags & KDA_G_FP32) ? static_cast<const float*>(f.g) : nullptr;
  p.beta = static_cast<const uint16_t*>(f.beta);
  p.dout = static_cast<const uint16_t*>(a->dout);
  p.A_log = f.A_log;
  p.dt_bias = f.dt_bias;
  p.lower_bound = f.lower_bound;
  p.scale = f.scale;
  p.gate_mode = (f.flags & KDA_GATE_UNSAFE) ? kGateUnsafe : (f.flags & KDA_GATE_LOGSPACE) ? kGateLogspace : kGateSafe;
  p.beta_prob = (f.flags & KDA_BETA_PROB) ? 1 : 0;
  p.l2norm = (f.flags & KDA_QK_L2NORM) ? 1 : 0;
  p.init = f.initial_state;
  p.init_bf16 = f.state_dtype == KDA_DTYPE_BF16 ? 1 : 0;
  p.dfinal = a->dfinal_state;
  p.cu = f.cu_seqlens;
  p.chunk_off = f.cu_seqlens ? reinterpret_cast<const int64_t*>(ws) : nullptr;
  p.N = f.N;
  p.T = f.T;
  p.H = H;
  p.NT = (f.T + kChunk - 1) / kChunk;
  p.nslots = slots;
  p.ws = reinterpret_cast<float*>(ws + round256(header));
  p.dq = a->dq;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dg = a->dg;
  p.dbeta = a->dbeta;
  p.dA_log = gate != KDA_GATE_LOGSPACE ? a->dA_log : nullptr;
  p.ddt_bias = gate != KDA_GATE_LOGSPACE ? a->ddt_bias : nullptr;
  p.dinit = a->dinitial_state;
  if (f.cu_seqlens) {
    // rows outside every chunk (all of them, if the bounds are inconsistent)
    // keep zero gradients
    const size_t tok = (size_t)rows * H * kHeadDim * sizeof(float);
    if (rows > 0) {
      chk(cudaMemsetAsync(a->dq, 0, tok, s));
      chk(cudaMemsetAsync(a->dk, 0, tok, s));
      chk(cudaMemsetAsync(a->dv, 0, tok, s));
      chk(cudaMemsetAsync(a->dg, 0, tok, s));
      chk(cudaMemsetAsync(a->dbeta, 0, (size_t)rows * H * sizeof(float), s));
    }
    launch_chunk_offsets(f.cu_seqlens, f.N, f.T, reinterpret_cast<int64_t*>(ws), status, s);
  }
  launch_bwd(p, s, events);
  if (!ok || cudaGetLastError() != cudaSuccess) return KDA_ERR_LAUNCH;
  return KDA_OK;
}
}  // namespace

extern "C" int kda_bwd(const kda_bwd_args* a, void* workspace, size_t workspace_bytes, void* stream_ptr) {
  return bwd_device(a, workspace, workspace_bytes, stream_ptr, nullptr);
}

extern "C" int kda_bwd_profiled(const kda_bwd_args* a, void* workspace, size_t workspace_bytes,
                                void* stream_ptr, void* const events[4]) {
  return bwd_device(a, workspace, workspace_bytes, stream_ptr, events);
}
