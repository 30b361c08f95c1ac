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
//     into the chunk's workspace item;
//  2. forward state pass, one CTA per (sequence, head, 16 value rows): walks the
//     chunks, storing S before each chunk and Unew (value rows are independent);
//  3. reverse state pass, same grid, chunks last to first from dfinal: stores
//     dS_C and dU of each chunk, then dinitial;
//  4. gradient products, one CTA per (chunk, head): dQg, dKhat, dKg, dP, dT, dgC, dv;
//  5. chunk gradients, one CTA per (chunk, head): dM, dG, dbeta, the pairwise
//     terms, the scalings, the cumulative sum, gate and norms: dq, dk, dg,
//     dbeta, and the chunk's parts of dA_log and dt_bias;
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
constexpr int kVb = 16;       // value rows per CTA of the state passes
constexpr int kRowBlocks = kD / kVb;

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
constexpr int kItemFloats = 98752;  // 395,008 bytes, a multiple of 256
static_assert(kItemPart + kD + 1 <= kItemFloats && kItemFloats % 64 == 0, "item layout");

constexpr int kStage = 16 * (kLs + kLd);  // GEMM staging floats
constexpr int kPrepFloats = 3 * kC * kLd + 3 * kC * kLs + 80 * kLd + kStage + kC;
constexpr int kGradFloats = 3 * kC * kLd + 2 * kC * kLs + 80 * kLd + kStage + 16 * kD + 4 * kC;
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
// z = g + dt_bias (logspace: g) of element (row, c)
__device__ __forceinline__ float gate_z(const BwdParams& p, int64_t row, int h, int c) {
  const float g = p.g32 ? p.g32[row * kD + c] : bf16_to_f(p.g[row * kD + c]);
  if (p.gate_mode == kGateLogspace || !p.dt_bias) return g;
  return g + p.dt_bias[h * kD + c];
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
// rows >= L are zero.  One warp per row, lane = 4 channels.
__device__ void load_rows(const BwdParams& p, const ChunkLoc& cl, int h, float* Kh, float* Qh,
                          float* vb, float* rq, float* rk) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = warp; t < kC; t += 8) {
    float q[4] = {0.f, 0.f, 0.f, 0.f}, k[4] = {0.f, 0.f, 0.f, 0.f};
    float b = 0.f;
    if (t < cl.L) {
      const int64_t row = (cl.t0 + t) * p.H + h;
      load4(p.q + row * kD + 4 * lane, q);
      load4(p.k + row * kD + 4 * lane, k);
      const float braw = bf16_to_f(p.beta[row]);
      b = p.beta_prob ? braw : 1.f / (1.f + expf(-braw));
    }
    float sq = 1.f, sk = 1.f;
    if (p.l2norm) {
      sq = rsqrtf(warp_sum(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]) + 1e-6f);
      sk = rsqrtf(warp_sum(k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3]) + 1e-6f);
    }
    st4(Qh + t * kLd + 4 * lane, q[0] * sq, q[1] * sq, q[2] * sq, q[3] * sq);
    st4(Kh + t * kLd + 4 * lane, k[0] * sk, k[1] * sk, k[2] * sk, k[3] * sk);
    if (lane == 0) {
      vb[t] = b;
      if (rq) rq[t] = sq;
      if (rk) rk[t] = sk;
    }
  }
}

// Gamma [64][kLd]: the in-chunk cumulative sums of the activated gate (a = 0 on
// rows >= L).  Ends with a barrier.
__device__ void gate_cumsum(const BwdParams& p, const ChunkLoc& cl, int h, float* Gm) {
  const float amul = gate_mul(p, h);
  for (int e = threadIdx.x; e < kC * kD; e += blockDim.x) {
    const int t = e >> 7, c = e & (kD - 1);
    float a = 0.f;
    if (t < cl.L) {
      float d1, d2;
      a = gate_a(p.gate_mode, gate_z(p, (cl.t0 + t) * p.H + h, h, c), amul, p.lower_bound, d1, d2);
    }
    Gm[t * kLd + c] = a;
  }
  __syncthreads();
  if (threadIdx.x < kD) {
    float acc = 0.f;
    for (int t = 0; t < kC; ++t) {
      acc += Gm[t * kLd + threadIdx.x];
      Gm[t * kLd + threadIdx.x] = acc;
    }
  }
  __syncthreads();
}

// ---- fp32 block GEMM (256 threads) ----
// Operand view: element (r, c) = p[r * ld + c] (fp32, or bf16 if b16); rows
// r >= rows read as zero.
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
__device__ __forceinline__ float opd_at(const Opd& o, int r, int c) {
  if (r >= o.rows) return 0.f;
  const int64_t i = (int64_t)r * o.ld + c;
  return o.b16 ? bf16_to_f(static_cast<const uint16_t*>(o.p)[i]) : static_cast<const float*>(o.p)[i];
}

// acc[4][BN / 16] += A (64 x kd) B (kd x BN), with A(m, k) = kAT ? a(k, m) : a(m, k)
// and B(k, n) = kBT ? b(n, k) : b(k, n); kd a multiple of 16.  Thread (ty =
// tid / 16, tx = tid % 16) owns rows 4 ty + i and columns 4 tx + j (j < 4) and
// 64 + 4 tx + j - 4 (j >= 4, BN = 128).  Staged through `stage` in
// 16-deep slices; begins and ends with a barrier.

template <int BN, bool kAT, bool kBT>
__device__ void gemm64(float (&acc)[4][BN / 16], const Opd& a, const Opd& b, int kd, float* stage) {
  constexpr int kBs = BN + 4;
  float* As = stage;             // [16][kLs]: As[k][m]
  float* Bs = stage + 16 * kLs;  // [16][kBs]: Bs[k][n]
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  for (int k0 = 0; k0 < kd; k0 += 16) {
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + 256 * i;
      if (kAT) {
        const int m = e & 63, k = e >> 6;
        As[k * kLs + m] = opd_at(a, k0 + k, m);
      } else {
        const int k = e & 15, m = e >> 4;
        As[k * kLs + m] = opd_at(a, m, k0 + k);
      }
    }
#pragma unroll
    for (int i = 0; i < BN / 16; ++i) {
      const int e = tid + 256 * i;
      if (kBT) {
        const int k = e & 15, n = e >> 4;
        Bs[k * kBs + n] = opd_at(b, n, k0 + k);
      } else {
        const int n = e % BN, k = e / BN;
        Bs[k * kBs + n] = opd_at(b, k0 + k, n);
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const float4 av = ld4(As + kk * kLs + 4 * ty);
      const float ar[4] = {av.x, av.y, av.z, av.w};
      float br[BN / 16];
      const float4 b0 = ld4(Bs + kk * kBs + 4 * tx);
      br[0] = b0.x;
      br[1] = b0.y;
      br[2] = b0.z;
      br[3] = b0.w;
      if constexpr (BN == 128) {
        const float4 b1 = ld4(Bs + kk * kBs + 64 + 4 * tx);
        br[4] = b1.x;
        br[5] = b1.y;
        br[6] = b1.z;
        br[7] = b1.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < BN / 16; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
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
__global__ void __launch_bounds__(256, 1) kda_bwd_prep_kernel(BwdParams p) {
  extern __shared__ __align__(16) float sm[];
  float* Kh = sm;
  float* Qh = Kh + kC * kLd;
  float* Gm = Qh + kC * kLd;
  float* Gs = Gm + kC * kLd;  // G, then T
  float* Ps = Gs + kC * kLs;
  float* Mi = Ps + kC * kLs;
  float* X = Mi + kC * kLs;   // [80][kLd]: Lk, Lq, R; then Kg
  float* stage = X + 80 * kLd;
  float* vb = stage + kStage;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t item = blockIdx.x, slot = item / p.H;
  const int h = (int)(item - slot * p.H);
  ChunkLoc cl;
  if (!locate(p, slot, cl)) return;
  float* it = p.ws + item * (int64_t)kItemFloats;

  load_rows(p, cl, h, Kh, Qh, vb, nullptr, nullptr);
  __syncthreads();
  gate_cumsum(p, cl, h, Gm);

  // G and P inside the 16-token diagonal blocks, pair by pair: one warp per pair
  for (int e = warp; e < 4 * 136; e += 8) {
    const int blk = e / 136, r = e - blk * 136;
    int ii = 0;
    while ((ii + 1) * (ii + 2) / 2 <= r) ++ii;
    const int jj = r - ii * (ii + 1) / 2;
    const int i = 16 * blk + ii, j = 16 * blk + jj;
    const float4 gi = ld4(Gm + i * kLd + 4 * lane), gj = ld4(Gm + j * kLd + 4 * lane);
    const float4 ki = ld4(Kh + i * kLd + 4 * lane), kj = ld4(Kh + j * kLd + 4 * lane);
    const float4 qi = ld4(Qh + i * kLd + 4 * lane);
    const float f0 = expf(gi.x - gj.x), f1 = expf(gi.y - gj.y), f2 = expf(gi.z - gj.z), f3 = expf(gi.w - gj.w);
    float sg = ki.x * kj.x * f0 + ki.y * kj.y * f1 + ki.z * kj.z * f2 + ki.w * kj.w * f3;
    float sp = qi.x * kj.x * f0 + qi.y * kj.y * f1 + qi.z * kj.z * f2 + qi.w * kj.w * f3;
    sg = warp_sum(sg);
    sp = warp_sum(sp);
    if (lane == 0) {
      Gs[i * kLs + j] = j < i ? sg : 0.f;
      Ps[i * kLs + j] = sp;
    }
  }
  // zero the upper triangles and the off-diagonal blocks' upper parts
  for (int e = tid; e < kC * kC; e += 256) {
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
    for (int e = tid; e < (32 + r) * 32; e += 256) {
      const int row = e >> 5, c = 4 * (e & 31);
      const float4 gr = ld4(Gm + r * kLd + c);
      if (row < 32) {  // Lk / Lq rows of block I
        const int ii = row & 15, i = r + ii;
        const float4 gi = ld4(Gm + i * kLd + c);
        const float l0 = expf(gi.x - gr.x), l1 = expf(gi.y - gr.y), l2 = expf(gi.z - gr.z), l3 = expf(gi.w - gr.w);
        const float4 x = ld4((row < 16 ? Kh : Qh) + i * kLd + c);
        st4((row < 16 ? Lk : Lq) + ii * kLd + c, x.x * l0, x.y * l1, x.z * l2, x.w * l3);
      } else {
        const int j = row - 32;
        const float4 gj = ld4(Gm + j * kLd + c);
        const float4 x = ld4(Kh + j * kLd + c);
        st4(R + j * kLd + c, x.x * expf(gr.x - gj.x), x.y * expf(gr.y - gj.y), x.z * expf(gr.z - gj.z),
            x.w * expf(gr.w - gj.w));
      }
    }
    __syncthreads();
    for (int e = tid; e < 16 * r; e += 256) {
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
  // Minv = (I + Diag(beta) G)^-1 by forward substitution: four lanes per column
  {
    const int col = warp * 8 + (lane >> 2), l = lane & 3;
    for (int i = 0; i < kC; ++i) {
      float s = 0.f;
      for (int m = col + l; m < i; m += 4) s = fmaf(Gs[i * kLs + m], Mi[m * kLs + col], s);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (l == 0) Mi[i * kLs + col] = i < col ? 0.f : (i == col ? 1.f : -vb[i] * s);
      __syncwarp();
    }
  }
  __syncthreads();
  // write G, P, Minv, gC, Qg, Khat, Kg; T = Minv Diag(beta) over G; Kg into X
  for (int e = tid; e < kC * kC; e += 256) {
    const int i = e >> 6, j = e & 63;
    it[kItemG + e] = Gs[i * kLs + j];
    it[kItemP + e] = Ps[i * kLs + j];
    it[kItemMi + e] = Mi[i * kLs + j];
  }
  __syncthreads();
  for (int e = tid; e < kC * kC; e += 256) {
    const int i = e >> 6, j = e & 63;
    Gs[i * kLs + j] = Mi[i * kLs + j] * vb[j];
  }
  for (int e = tid; e < kC * 32; e += 256) {
    const int t = e >> 5, c = 4 * (e & 31);
    const float4 gt = ld4(Gm + t * kLd + c), gl = ld4(Gm + (kC - 1) * kLd + c);
    const float4 kx = ld4(Kh + t * kLd + c), qx = ld4(Qh + t * kLd + c);
    const float e0 = expf(gt.x), e1 = expf(gt.y), e2 = expf(gt.z), e3 = expf(gt.w);
    st4(it + kItemQg + t * kD + c, qx.x * e0, qx.y * e1, qx.z * e2, qx.w * e3);
    st4(it + kItemKg + t * kD + c, kx.x * e0, kx.y * e1, kx.z * e2, kx.w * e3);
    st4(X + t * kLd + c, kx.x * e0, kx.y * e1, kx.z * e2, kx.w * e3);
    st4(it + kItemKh + t * kD + c, kx.x * expf(gl.x - gt.x), kx.y * expf(gl.y - gt.y), kx.z * expf(gl.z - gt.z),
        kx.w * expf(gl.w - gt.w));
  }
  if (tid < kD) it[kItemGC + tid] = expf(Gm[(kC - 1) * kLd + tid]);
  // W = T Kg, U = T V
  const int ty = tid >> 4, tx = tid & 15;
  {
    float acc[4][8];
    zero_acc(acc);
    gemm64<128, false, false>(acc, opd(Gs, kLs, kC), opd(X, kLd, kC), kC, stage);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float* dst = it + kItemW + (4 * ty + i) * kD;
      st4(dst + 4 * tx, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      st4(dst + 64 + 4 * tx, acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
  }
  {
    float acc[4][8];
    zero_acc(acc);
    gemm64<128, false, false>(acc, opd(Gs, kLs, kC), opd(p.v + (cl.t0 * p.H + h) * kD, p.H * kD, cl.L, 1), kC,
                              stage);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float* dst = it + kItemU + (4 * ty + i) * kD;
      st4(dst + 4 * tx, acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      st4(dst + 64 + 4 * tx, acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
    }
  }
}

// ==== 2. forward state pass ====
// CTA = (sequence, head, 16 value rows v0 ..).  Product 1 (Unew = U - W S^T,
// 64 x 16 over 128 channels): lane = (2 tokens, 4 value rows, channel half),
// halves combined by a shuffle.  Product 2 (S = S Diag(gC) + Unew^T Khat, 16 x
// 128 over 64 tokens): thread = (4 value rows, 8 channels, token quarter),
// quarters combined by shuffles; every quarter keeps the full result.
__global__ void __launch_bounds__(256) kda_bwd_fwd_state_kernel(BwdParams p) {
  __shared__ __align__(16) float Ss[kVb * kLd];
  __shared__ __align__(16) float Un[kC * kVb];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x / kRowBlocks;
  const int v0 = kVb * (int)(blockIdx.x - unit * kRowBlocks);
  const int64_t n = unit / p.H;
  const int h = (int)(unit - n * p.H);
  // product-2 ownership
  const int tq = lane & 3, co = ((warp & 1) << 3) | (lane >> 2), vq = warp >> 1;
  float s[4][8];
  {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD + 8 * co;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float x = 0.f;
        if (p.init) {
          const int64_t e = base + (int64_t)i * kD + j;
          x = p.init_bf16 ? bf16_to_f(static_cast<const uint16_t*>(p.init)[e])
                          : static_cast<const float*>(p.init)[e];
        }
        s[i][j] = x;
      }
  }
  if (tq == 0)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(Ss + (4 * vq + i) * kLd + 8 * co, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(Ss + (4 * vq + i) * kLd + 8 * co + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  // product-1 ownership
  const int ch = lane & 1, pv = (lane >> 1) & 3, pt = 8 * warp + 2 * (lane >> 3);
  int64_t first, count;
  seq_chunks(p, n, first, count);
  for (int64_t ci = 0; ci < count; ++ci) {
    float* it = p.ws + ((first + ci) * p.H + h) * (int64_t)kItemFloats;
    __syncthreads();  // Ss holds S before this chunk
    if (tq == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = it + kItemS0 + (v0 + 4 * vq + i) * kD + 8 * co;
        st4(d, s[i][0], s[i][1], s[i][2], s[i][3]);
        st4(d + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
      }
    {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const float* W0 = it + kItemW + pt * kD;
#pragma unroll 4
      for (int c = 64 * ch; c < 64 * ch + 64; c += 4) {
        const float4 w0 = ld4(W0 + c), w1 = ld4(W0 + kD + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 sv = ld4(Ss + (4 * pv + i) * kLd + c);
          acc[0][i] += w0.x * sv.x + w0.y * sv.y + w0.z * sv.z + w0.w * sv.w;
          acc[1][i] += w1.x * sv.x + w1.y * sv.y + w1.z * sv.z + w1.w * sv.w;
        }
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[r][i] += __shfl_xor_sync(0xffffffffu, acc[r][i], 1);
      if (ch == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float* u = it + kItemU + (pt + r) * kD + v0 + 4 * pv;
          const float4 uu = ld4(u);
          const float n0 = uu.x - acc[r][0], n1 = uu.y - acc[r][1], n2 = uu.z - acc[r][2], n3 = uu.w - acc[r][3];
          st4(u, n0, n1, n2, n3);
          st4(Un + (pt + r) * kVb + 4 * pv, n0, n1, n2, n3);
        }
      }
    }
    __syncthreads();  // Unew complete; Ss no longer read
    {
      float acc[4][8];
      zero_acc(acc);
      const float* K0 = it + kItemKh + 8 * co;
#pragma unroll 4
      for (int t = 16 * tq; t < 16 * tq + 16; ++t) {
        const float4 u = ld4(Un + t * kVb + 4 * vq);
        const float4 k0 = ld4(K0 + t * kD), k1 = ld4(K0 + t * kD + 4);
        const float ur[4] = {u.x, u.y, u.z, u.w}, kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(ur[i], kr[j], acc[i][j]);
      }
      const float4 g0 = ld4(it + kItemGC + 8 * co), g1 = ld4(it + kItemGC + 8 * co + 4);
      const float gr[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = acc[i][j];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          s[i][j] = fmaf(s[i][j], gr[j], x);
        }
      if (tq == 0)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          st4(Ss + (4 * vq + i) * kLd + 8 * co, s[i][0], s[i][1], s[i][2], s[i][3]);
          st4(Ss + (4 * vq + i) * kLd + 8 * co + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
        }
    }
  }
}

// ==== 3. reverse state pass ====
// Same grid and ownership as the forward pass.  Product A (dU = scale P^T dO +
// Khat dS^T, 64 x 16): lane = (2 tokens, 4 value rows, half of the 64 tokens j
// and of the 128 channels).  Product B (dS = dS Diag(gC) + scale dO^T Qg -
// dU^T W, 16 x 128 over 64 tokens).
__global__ void __launch_bounds__(256) kda_bwd_rev_state_kernel(BwdParams p) {
  __shared__ __align__(16) float Ds[kVb * kLd];
  __shared__ __align__(16) float Os[kC * kVb];   // scale dO, this CTA's value columns
  __shared__ __align__(16) float Us[kC * kVb];   // dU
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t unit = blockIdx.x / kRowBlocks;
  const int v0 = kVb * (int)(blockIdx.x - unit * kRowBlocks);
  const int64_t n = unit / p.H;
  const int h = (int)(unit - n * p.H);
  const int tq = lane & 3, co = ((warp & 1) << 3) | (lane >> 2), vq = warp >> 1;
  float s[4][8];
  {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD + 8 * co;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) s[i][j] = p.dfinal ? p.dfinal[base + (int64_t)i * kD + j] : 0.f;
  }
  if (tq == 0)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(Ds + (4 * vq + i) * kLd + 8 * co, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(Ds + (4 * vq + i) * kLd + 8 * co + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  const int ch = lane & 1, pv = (lane >> 1) & 3, pt = 8 * warp + 2 * (lane >> 3);
  int64_t first, count;
  seq_chunks(p, n, first, count);
  for (int64_t ci = count - 1; ci >= 0; --ci) {
    const int64_t slot = first + ci;
    float* it = p.ws + (slot * p.H + h) * (int64_t)kItemFloats;
    const int64_t t0 = p.cu ? p.cu[n] + ci * kC : n * p.T + ci * kC;
    const int L = (int)min((int64_t)kC, (p.cu ? p.cu[n + 1] : (n + 1) * p.T) - t0);
    __syncthreads();  // Ds holds dS_C; Os, Us free
    for (int e = tid; e < kC * kVb; e += 256) {
      const int t = e >> 4, v = e & 15;
      Os[e] = t < L ? p.scale * bf16_to_f(p.dout[((t0 + t) * p.H + h) * kD + v0 + v]) : 0.f;
    }
    if (tq == 0)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float* d = it + kItemDS + (v0 + 4 * vq + i) * kD + 8 * co;
        st4(d, s[i][0], s[i][1], s[i][2], s[i][3]);
        st4(d + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
      }
    __syncthreads();
    {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const float* K0 = it + kItemKh + pt * kD;
#pragma unroll 4
      for (int c = 64 * ch; c < 64 * ch + 64; c += 4) {
        const float4 k0 = ld4(K0 + c), k1 = ld4(K0 + kD + c);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 d = ld4(Ds + (4 * pv + i) * kLd + c);
          acc[0][i] += k0.x * d.x + k0.y * d.y + k0.z * d.z + k0.w * d.w;
          acc[1][i] += k1.x * d.x + k1.y * d.y + k1.z * d.z + k1.w * d.w;
        }
      }
      const float* P0 = it + kItemP + pt;
#pragma unroll 4
      for (int j = 32 * ch; j < 32 * ch + 32; ++j) {
        const float2 pj = *reinterpret_cast<const float2*>(P0 + j * kC);
        const float4 o = ld4(Os + j * kVb + 4 * pv);
        acc[0][0] += pj.x * o.x;
        acc[0][1] += pj.x * o.y;
        acc[0][2] += pj.x * o.z;
        acc[0][3] += pj.x * o.w;
        acc[1][0] += pj.y * o.x;
        acc[1][1] += pj.y * o.y;
        acc[1][2] += pj.y * o.z;
        acc[1][3] += pj.y * o.w;
      }
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[r][i] += __shfl_xor_sync(0xffffffffu, acc[r][i], 1);
      if (ch == 0) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          st4(it + kItemDU + (pt + r) * kD + v0 + 4 * pv, acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
          st4(Us + (pt + r) * kVb + 4 * pv, acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
        }
      }
    }
    __syncthreads();
    {
      float acc[4][8];
      zero_acc(acc);
      const float* Q0 = it + kItemQg + 8 * co;
      const float* W0 = it + kItemW + 8 * co;
#pragma unroll 2
      for (int t = 16 * tq; t < 16 * tq + 16; ++t) {
        const float4 o = ld4(Os + t * kVb + 4 * vq), u = ld4(Us + t * kVb + 4 * vq);
        const float4 q0 = ld4(Q0 + t * kD), q1 = ld4(Q0 + t * kD + 4);
        const float4 w0 = ld4(W0 + t * kD), w1 = ld4(W0 + t * kD + 4);
        const float orr[4] = {o.x, o.y, o.z, o.w}, ur[4] = {u.x, u.y, u.z, u.w};
        const float qr[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const float wr[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(orr[i], qr[j], fmaf(-ur[i], wr[j], acc[i][j]));
      }
      const float4 g0 = ld4(it + kItemGC + 8 * co), g1 = ld4(it + kItemGC + 8 * co + 4);
      const float gr[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float x = acc[i][j];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          s[i][j] = fmaf(s[i][j], gr[j], x);
        }
      if (tq == 0)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          st4(Ds + (4 * vq + i) * kLd + 8 * co, s[i][0], s[i][1], s[i][2], s[i][3]);
          st4(Ds + (4 * vq + i) * kLd + 8 * co + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
        }
    }
  }
  if (p.dinit && tq == 0) {
    const int64_t base = (unit * kD + v0 + 4 * vq) * kD + 8 * co;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st4(p.dinit + base + (int64_t)i * kD, s[i][0], s[i][1], s[i][2], s[i][3]);
      st4(p.dinit + base + (int64_t)i * kD + 4, s[i][4], s[i][5], s[i][6], s[i][7]);
    }
  }
}

// ==== 4. gradient products ====
__global__ void __launch_bounds__(256) kda_bwd_prod_kernel(BwdParams p) {
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
  gemm64<128, false, false>(acc, dO, S0, kD, stage);
  store128(it + kItemQg, acc, p.scale);
  // dW = -dU S (shared memory)
  zero_acc(acc);
  gemm64<128, false, false>(acc, dU, S0, kD, stage);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* d = dWs + (4 * ty + i) * kLd;
    st4(d + 4 * tx, -acc[i][0], -acc[i][1], -acc[i][2], -acc[i][3]);
    st4(d + 64 + 4 * tx, -acc[i][4], -acc[i][5], -acc[i][6], -acc[i][7]);
  }
  // dKhat = Unew dS_C
  zero_acc(acc);
  gemm64<128, false, false>(acc, Un, dS, kD, stage);
  store128(it + kItemKh, acc, 1.f);
  // dgC = colsum(S . dS_C)
  if (tid < kD) {
    float x = 0.f;
    for (int v = 0; v < kD; ++v) x = fmaf(it[kItemS0 + v * kD + tid], it[kItemDS + v * kD + tid], x);
    it[kItemDGC + tid] = x;
  }
  // dP = scale dO Unew^T (s <= t)
  {
    float a2[4][4];
    zero_acc(a2);
    gemm64<64, false, true>(a2, dO, Un, kD, stage);
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
    gemm64<64, false, true>(a2, dU, Vv, kD, stage);
    gemm64<64, false, true>(a2, opd(dWs, kLd, kC), Kg, kD, stage);
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
  gemm64<128, true, false>(acc, Mi, dU, kC, stage);
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
  gemm64<128, true, false>(acc, Mi, opd(dWs, kLd, kC), kC, stage);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float* d = it + kItemW + (4 * ty + i) * kD;
    st4(d + 4 * tx, bt[i] * acc[i][0], bt[i] * acc[i][1], bt[i] * acc[i][2], bt[i] * acc[i][3]);
    st4(d + 64 + 4 * tx, bt[i] * acc[i][4], bt[i] * acc[i][5], bt[i] * acc[i][6], bt[i] * acc[i][7]);
  }
}

// ==== 5. chunk gradients ====
// Thread (ty = tid / 16, tx = tid % 16) accumulates dq_hat, dk_hat and dGamma
// of rows 16 m + ty (m = 0..3), channels 8 tx .. 8 tx + 7, in registers.
__global__ void __launch_bounds__(256, 1) kda_bwd_grad_kernel(BwdParams p) {
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
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int64_t item = blockIdx.x, slot = item / p.H;
  const int h = (int)(item - slot * p.H);
  ChunkLoc cl;
  if (!locate(p, slot, cl)) return;
  float* it = p.ws + item * (int64_t)kItemFloats;

  load_rows(p, cl, h, Kh, Qh, vb, rq, rk);
  __syncthreads();
  gate_cumsum(p, cl, h, Gm);

  // ---- dM = -Minv^T (dT Diag(beta)) Minv^T, dA, dG, dbeta ----
  {
    float* Xa = X;             // dT Diag(beta) [64][kLs]
    float* Xb = X + kC * kLs;  // Minv^T dT Diag(beta)
    for (int e = tid; e < kC * kC; e += 256) {
      const int i = e >> 6, j = e & 63;
      Xa[i * kLs + j] = it[kItemDT + e] * vb[j];
      dPs[i * kLs + j] = it[kItemP + e];
    }
    if (tid < kC) {  // (Minv^T dT)_tt
      float x = 0.f;
      for (int j = tid; j < kC; ++j) x = fmaf(it[kItemMi + j * kC + tid], it[kItemDT + j * kC + tid], x);
      dbv[tid] = x;
    }
    float a2[4][4];
    zero_acc(a2);
    gemm64<64, true, false>(a2, opd(it + kItemMi, kC, kC), opd(Xa, kLs, kC), kC, stage);
#pragma unroll
    for (int i = 0; i < 4; ++i) st4(Xb + (4 * ty + i) * kLs + 4 * tx, a2[i][0], a2[i][1], a2[i][2], a2[i][3]);
    zero_acc(a2);
    gemm64<64, false, true>(a2, opd(Xb, kLs, kC), opd(it + kItemMi, kC, kC), kC, stage);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = 4 * ty + i;
      float d[4], gsum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = 4 * tx + j;
        const float dA = s < t ? -a2[i][j] : 0.f;
        gsum = fmaf(dA, it[kItemG + t * kC + s], gsum);
        d[j] = vb[t] * dA;
      }
      st4(dGs + t * kLs + 4 * tx, d[0], d[1], d[2], d[3]);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, o);
      if (tx == 0) dbv[t] += gsum;
    }
  }
  __syncthreads();

  float aQ[4][8], aK[4][8], aG[4][8];
  // ---- the scalings: Qg = q e^Gamma, Kg = k e^Gamma, Khat = k e^{Gamma_C - Gamma} ----
  {
    float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int t = 16 * m + ty;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = 8 * tx + j;
        const float gt = Gm[t * kLd + c], e = expf(gt), ec = expf(Gm[(kC - 1) * kLd + c] - gt);
        const float qh = Qh[t * kLd + c], kh = Kh[t * kLd + c];
        const float dqg = it[kItemQg + t * kD + c], dkg = it[kItemW + t * kD + c], dkh = it[kItemKh + t * kD + c];
        aQ[m][j] = dqg * e;
        aK[m][j] = dkg * e + dkh * ec;
        aG[m][j] = dqg * qh * e + dkg * kh * e - dkh * kh * ec;
        cs[j] += dkh * kh * ec;
      }
    }
    st4(part + ty * kD + 8 * tx, cs[0], cs[1], cs[2], cs[3]);
    st4(part + ty * kD + 8 * tx + 4, cs[4], cs[5], cs[6], cs[7]);
  }
  // ---- G and P inside the diagonal blocks, pair by pair ----
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int t = 16 * m + ty;
    float gt[8], kt[8], qt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      gt[j] = Gm[t * kLd + 8 * tx + j];
      kt[j] = Kh[t * kLd + 8 * tx + j];
      qt[j] = Qh[t * kLd + 8 * tx + j];
    }
    const float dpd = dPs[t * kLs + t];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      aQ[m][j] = fmaf(dpd, kt[j], aQ[m][j]);
      aK[m][j] = fmaf(dpd, qt[j], aK[m][j]);
    }
    for (int s = 16 * m; s < 16 * m + 16; ++s) {
      if (s == t) continue;
      float gs[8], ks[8], qs[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        gs[j] = Gm[s * kLd + 8 * tx + j];
        ks[j] = Kh[s * kLd + 8 * tx + j];
        qs[j] = Qh[s * kLd + 8 * tx + j];
      }
      if (s < t) {  // t takes the role of the later token
        const float dg = dGs[t * kLs + s], dp = dPs[t * kLs + s];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float f = expf(gt[j] - gs[j]) * ks[j];
          aK[m][j] = fmaf(dg, f, aK[m][j]);
          aQ[m][j] = fmaf(dp, f, aQ[m][j]);
          aG[m][j] = fmaf(dg * kt[j] + dp * qt[j], f, aG[m][j]);
        }
      } else {  // t is the earlier token
        const float dg = dGs[s * kLs + t], dp = dPs[s * kLs + t];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float w = (dg * ks[j] + dp * qs[j]) * expf(gs[j] - gt[j]);
          aK[m][j] = fmaf(w, 1.f, aK[m][j]);
          aG[m][j] = fmaf(-w, kt[j], aG[m][j]);
        }
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
    for (int e = tid; e < (32 + r) * 32; e += 256) {
      const int row = e >> 5, c = 4 * (e & 31);
      const float4 gr = ld4(Gm + r * kLd + c);
      if (row < 32) {
        const int ii = row & 15, i = r + ii;
        const float4 gi = ld4(Gm + i * kLd + c);
        const float4 x = ld4((row < 16 ? Kh : Qh) + i * kLd + c);
        st4((row < 16 ? Lk : Lq) + ii * kLd + c, x.x * expf(gi.x - gr.x), x.y * expf(gi.y - gr.y),
            x.z * expf(gi.z - gr.z), x.w * expf(gi.w - gr.w));
      } else {
        const int j = row - 32;
        const float4 gj = ld4(Gm + j * kLd + c);
        const float4 x = ld4(Kh + j * kLd + c);
        st4(R + j * kLd + c, x.x * expf(gr.x - gj.x), x.y * expf(gr.y - gj.y), x.z * expf(gr.z - gj.z),
            x.w * expf(gr.w - gj.w));
      }
    }
    __syncthreads();
    {  // rows of block I (t = r + ty): X_G = dG R, X_P = dP R over s < r
      const int t = r + ty;
      float xg[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, xp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int s = 0; s < r; ++s) {
        const float dg = dGs[t * kLs + s], dp = dPs[t * kLs + s];
        const float4 r0 = ld4(R + s * kLd + 8 * tx), r1 = ld4(R + s * kLd + 8 * tx + 4);
        const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          xg[j] = fmaf(dg, rr[j], xg[j]);
          xp[j] = fmaf(dp, rr[j], xp[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = 8 * tx + j;
        const float l = expf(Gm[t * kLd + c] - Gm[r * kLd + c]);
        aK[I][j] = fmaf(l, xg[j], aK[I][j]);
        aQ[I][j] = fmaf(l, xp[j], aQ[I][j]);
        aG[I][j] = fmaf(l, Kh[t * kLd + c] * xg[j] + Qh[t * kLd + c] * xp[j], aG[I][j]);
      }
    }
#pragma unroll
    for (int m = 0; m < I; ++m) {  // rows s = 16 m + ty < r: Y = dG^T Lk + dP^T Lq over block I
      const int s = 16 * m + ty;
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int ii = 0; ii < 16; ++ii) {
        const float dg = dGs[(r + ii) * kLs + s], dp = dPs[(r + ii) * kLs + s];
        const float4 k0 = ld4(Lk + ii * kLd + 8 * tx), k1 = ld4(Lk + ii * kLd + 8 * tx + 4);
        const float4 q0 = ld4(Lq + ii * kLd + 8 * tx), q1 = ld4(Lq + ii * kLd + 8 * tx + 4);
        const float kr[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        const float qr[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = fmaf(dg, kr[j], fmaf(dp, qr[j], y[j]));
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int c = 8 * tx + j;
        const float rr = R[s * kLd + c];                       // k_s e^{Gamma_r - Gamma_s}
        const float e = expf(Gm[r * kLd + c] - Gm[s * kLd + c]);
        aK[m][j] = fmaf(e, y[j], aK[m][j]);
        aG[m][j] = fmaf(-rr, y[j], aG[m][j]);
      }
    }
  }
  __syncthreads();
  // ---- dGamma -> da by the reverse cumulative sum ----
  float* Dg = X;  // [64][kLd]
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    float* d = Dg + (16 * m + ty) * kLd + 8 * tx;
    st4(d, aG[m][0], aG[m][1], aG[m][2], aG[m][3]);
    st4(d + 4, aG[m][4], aG[m][5], aG[m][6], aG[m][7]);
  }
  __syncthreads();
  if (tid < kD) {
    float x = it[kItemDGC + tid] * expf(Gm[(kC - 1) * kLd + tid]);
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
  const float amul = gate_mul(p, h);
  float pdt[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, pal = 0.f;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int t = 16 * m + ty;
    const bool live = t < cl.L;
    const int64_t row = (cl.t0 + (live ? t : 0)) * p.H + h;
    float xq = 0.f, xk = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      xq = fmaf(Qh[t * kLd + 8 * tx + j], aQ[m][j], xq);
      xk = fmaf(Kh[t * kLd + 8 * tx + j], aK[m][j], xk);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      xq += __shfl_xor_sync(0xffffffffu, xq, o);
      xk += __shfl_xor_sync(0xffffffffu, xk, o);
    }
    if (!live) continue;
    float dq[8], dk[8], dz[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = 8 * tx + j;
      if (p.l2norm) {
        dq[j] = rq[t] * (aQ[m][j] - Qh[t * kLd + c] * xq);
        dk[j] = rk[t] * (aK[m][j] - Kh[t * kLd + c] * xk);
      } else {
        dq[j] = aQ[m][j];
        dk[j] = aK[m][j];
      }
      float dadz, dadA;
      gate_a(p.gate_mode, gate_z(p, row, h, c), amul, p.lower_bound, dadz, dadA);
      const float da = Dg[t * kLd + c];
      dz[j] = da * dadz;
      pdt[j] += dz[j];
      pal = fmaf(da, dadA, pal);
    }
    float* o = p.dq + row * kD + 8 * tx;
    st4(o, dq[0], dq[1], dq[2], dq[3]);
    st4(o + 4, dq[4], dq[5], dq[6], dq[7]);
    o = p.dk + row * kD + 8 * tx;
    st4(o, dk[0], dk[1], dk[2], dk[3]);
    st4(o + 4, dk[4], dk[5], dk[6], dk[7]);
    o = p.dg + row * kD + 8 * tx;
    st4(o, dz[0], dz[1], dz[2], dz[3]);
    st4(o + 4, dz[4], dz[5], dz[6], dz[7]);
  }
  if (tid < cl.L) {
    float db = dbv[tid];
    if (!p.beta_prob) db *= vb[tid] * (1.f - vb[tid]);
    p.dbeta[(cl.t0 + tid) * p.H + h] = db;
  }
  // the chunk's parts of dt_bias and A_log, summed in a fixed order
  __syncthreads();
  st4(part + ty * kD + 8 * tx, pdt[0], pdt[1], pdt[2], pdt[3]);
  st4(part + ty * kD + 8 * tx + 4, pdt[4], pdt[5], pdt[6], pdt[7]);
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
    for (int w = 0; w < 8; ++w) x += X[w];
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
  const unsigned units = (unsigned)(p.N * p.H * kRowBlocks);
  if (items) kda_bwd_prep_kernel<<<items, 256, kPrepFloats * 4, s>>>(p);
  kda_bwd_fwd_state_kernel<<<units, 256, 0, s>>>(p);
  mark(1);
  kda_bwd_rev_state_kernel<<<units, 256, 0, s>>>(p);
  mark(2);
  if (items) {
    kda_bwd_prod_kernel<<<items, 256, kProdFloats * 4, s>>>(p);
    kda_bwd_grad_kernel<<<items, 256, kGradFloats * 4, s>>>(p);
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
