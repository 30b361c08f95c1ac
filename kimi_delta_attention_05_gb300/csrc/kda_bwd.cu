// Backward pass of the KDA forward (the "chunk_bwd" stage of the fla-kda code
// map, here in token-recurrent form): gradients of L = <out, dout> +
// <final_state, dfinal_state> with respect to q, k, v, g, beta, A_log,
// dt_bias and the initial state.
//
// Per value row s of the state (row = value index, a vector over the 128 key
// channels) the forward step of token t is
//     s' = s Diag(D),  D = exp(a_t);   u = v_t[row] - s' . k;   s = s' + beta u k
//     o_t[row] = scale s . q
// (k, q L2-normalised if asked).  Rows evolve independently; the reverse step,
// given ds = dL/ds after token t and do = dout_t[row], is
//     ds += scale do q;          dq  += scale do s
//     dsk = ds . k;              dbeta += u dsk;     du = beta dsk
//     dk += beta u ds - du s';   dv_t[row] = du
//     ds' = ds - du k;           dD += ds' (x) s_prev;   ds = ds' Diag(D)
// and dL/d(initial state) is ds after the first token.  dq, dk, dD and dbeta
// are sums over the 128 rows.
//
// The 128 value rows of a (sequence, head) are split over R CTAs ("row
// blocks", R a power of two chosen per call so that the grid covers the GPU:
// 16 / R warps of 8 value rows each, lane = 4 key channels).  Three launches:
//  1. checkpoints: the forward recurrence of the CTA's rows, a block of kBwdBlock
//     tokens at a time (the block's normalised k, D, beta and v staged in shared memory),
//     storing the state (fp32) at the start of every block;
//  2. reverse walk: per block (last to first) the block's k, q (normalised),
//     D, beta, v and dout are staged in shared memory; for each token, last to
//     first, the state before it is recomputed from the block's checkpoint with
//     the same step (bit-identical to pass 1), the reverse step is applied, and
//     the per-row terms of dq, dk, dD, dbeta are summed over the CTA's rows in
//     shared memory into the row block's part of a per-token-head record;
//  3. finalize, one warp per (run of 64 packed token rows, head): the R parts
//     of each record are summed in row-block order, and the L2-norm, gate and
//     sigmoid derivatives turn them into dq, dk, dg, dbeta; the sums over tokens
//     give dA_log and dt_bias (float atomics, one per channel per run).
#include <atomic>

#include "../../include/kda.h"
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

constexpr int kBwdBlock = 8;                   // tokens per checkpoint
constexpr int kBwdWarps = 16;                  // x 8 value rows = 128
constexpr int kBwdThreads = 32 * kBwdWarps;
// record of a token-head: dq_hat, dk_hat, dD (128 each), dbeta, padded to a
// multiple of four floats so that every 128-float part starts 16-byte aligned
// (the parts are read and written as float4)
constexpr int kBwdRec = 3 * kHeadDim + 4;
constexpr int kBwdRecBeta = 3 * kHeadDim;      // index of dbeta in a record

__device__ __forceinline__ float rcp_fast_b(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float warp_sum_b(float x) {
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

// Per-head gate constants.
struct GateC {
  float amul, lb;
  float dtb[4];
};

// The token's forward quantities on this lane's key channels c0 .. c0 + 3:
// normalised k, q, the decay D = exp(a) and beta.  One warp computes one
// token; every warp and every pass computes them with this same code.
template <int kGate, bool kL2>
__device__ __forceinline__ void token_inputs(const BwdParams& p, int64_t row, int c0, const GateC& gc,
                                             float (&k)[4], float (&q)[4], float (&D)[4], float& beta) {
  float g[4];
  load4(p.q + row * kHeadDim + c0, q);
  load4(p.k + row * kHeadDim + c0, k);
  if (p.g32) {
    const float4 x = *reinterpret_cast<const float4*>(p.g32 + row * kHeadDim + c0);
    g[0] = x.x;
    g[1] = x.y;
    g[2] = x.z;
    g[3] = x.w;
  } else {
    load4(p.g + row * kHeadDim + c0, g);
  }
  const float braw = bf16_to_f(p.beta[row]);
  beta = p.beta_prob ? braw : rcp_fast_b(1.0f + ex2(-braw * kLog2e));
  if (kL2) {
    const float rq = rsqrtf(warp_sum_b(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]) + 1e-6f);
    const float rk = rsqrtf(warp_sum_b(k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3]) + 1e-6f);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      q[c] *= rq;
      k[c] *= rk;
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float z = kGate == kGateLogspace ? g[c] : g[c] + gc.dtb[c];
    float d;
    if (kGate == kGateLogspace) d = ex2(z * kLog2e);
    else if (kGate == kGateUnsafe) d = ex2(-gc.amul * lg2(1.0f + ex2(z * kLog2e)));
    else d = ex2(gc.lb * kLog2e * rcp_fast_b(1.0f + ex2(-gc.amul * kLog2e * z)));
    D[c] = d;
  }
}

// One forward step of 8 rows (this lane's 4 channels each).
__device__ __forceinline__ void fwd_step(float (&S)[8][4], const float (&k)[4], const float (&D)[4],
                                         float beta, const float (&v)[8]) {
  float pr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    pr[i] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      S[i][c] *= D[c];
      pr[i] += S[i][c] * k[c];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) pr[i] = warp_sum_b(pr[i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float w = beta * (v[i] - pr[i]);
#pragma unroll
    for (int c = 0; c < 4; ++c) S[i][c] += w * k[c];
  }
}

__device__ __forceinline__ GateC gate_consts(const BwdParams& p, int h, int c0) {
  GateC gc;
  gc.amul = (p.A_log && p.gate_mode != kGateLogspace) ? expf(p.A_log[h]) : 1.0f;
  gc.lb = p.lower_bound;
  for (int c = 0; c < 4; ++c)
    gc.dtb[c] = (p.dt_bias && p.gate_mode != kGateLogspace) ? p.dt_bias[h * kHeadDim + c0 + c] : 0.f;
  return gc;
}

// Sequence bounds of unit (n, h); a sequence whose cu_seqlens bounds leave
// [0, T] or decrease is skipped (its token gradients stay zero, dinitial =
// dfinal) and the status word is set.
__device__ __forceinline__ void seq_bounds(const BwdParams& p, int64_t n, int64_t& bos, int64_t& eos) {
  bos = p.cu ? p.cu[n] : n * p.T;
  eos = p.cu ? p.cu[n + 1] : bos + p.T;
  if (p.cu) {
    const bool inside = bos >= 0 && eos >= bos && eos <= p.T;
    const bool bad = !inside || (n == 0 && bos != 0) || (n == p.N - 1 && eos != p.T);
    if (bad && threadIdx.x == 0 && p.status) atomicExch(p.status, KDA_ERR_BAD_SEQLENS);
    if (!inside) eos = bos;
  }
}

// ---- pass 1: checkpoints ----
template <int kGate, bool kL2>
__global__ void __launch_bounds__(kBwdThreads) kda_bwd_ckpt_kernel(BwdParams p, int rsplit) {
  __shared__ float sk[kBwdBlock][kHeadDim], sd[kBwdBlock][kHeadDim], sv[kBwdBlock][kHeadDim];
  __shared__ float sb[kBwdBlock];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t H = p.H;
  const int64_t unit = blockIdx.x / rsplit;
  const int rb = (int)(blockIdx.x - unit * rsplit);
  const int64_t n = unit / H;
  const int h = (int)(unit - n * H);
  int64_t bos, eos;
  seq_bounds(p, n, bos, eos);
  const int c0 = 4 * lane, r0 = 8 * (warp + nw * rb);
  const int64_t sbase = unit * (int64_t)(kHeadDim * kHeadDim);
  const GateC gc = gate_consts(p, h, c0);
  float S[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t off = sbase + (int64_t)(r0 + i) * kHeadDim + c0;
    if (!p.init) {
      S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
    } else if (p.init_bf16) {
      load4(reinterpret_cast<const uint16_t*>(p.init) + off, S[i]);
    } else {
      const float4 x = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.init) + off);
      S[i][0] = x.x;
      S[i][1] = x.y;
      S[i][2] = x.z;
      S[i][3] = x.w;
    }
  }
  float* ck = p.ckpt + (h * p.nslots + bos / kBwdBlock + n) * (int64_t)(kHeadDim * kHeadDim);
  const int64_t nblk = (eos - bos + kBwdBlock - 1) / kBwdBlock;
  for (int64_t blk = 0; blk < nblk; ++blk) {
    const int64_t t_lo = bos + blk * kBwdBlock;
    const int nt = (int)min((int64_t)kBwdBlock, eos - t_lo);
    __syncthreads();  // the previous block's staging is no longer read
    for (int j = warp; j < nt; j += nw) {  // warp w stages tokens w, w + nw, ...
      const int64_t row = (t_lo + j) * H + h;
      float k[4], q[4], D[4], beta, vv[4];
      token_inputs<kGate, kL2>(p, row, c0, gc, k, q, D, beta);
      load4(p.v + row * kHeadDim + c0, vv);
      *reinterpret_cast<float4*>(&sk[j][c0]) = make_float4(k[0], k[1], k[2], k[3]);
      *reinterpret_cast<float4*>(&sd[j][c0]) = make_float4(D[0], D[1], D[2], D[3]);
      *reinterpret_cast<float4*>(&sv[j][c0]) = make_float4(vv[0], vv[1], vv[2], vv[3]);
      if (lane == 0) sb[j] = beta;
    }
    __syncthreads();
    float* dst = ck + blk * (int64_t)(kHeadDim * kHeadDim);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(dst + (r0 + i) * kHeadDim + c0) = make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    for (int j = 0; j < nt; ++j) {
      const float4 kk = *reinterpret_cast<const float4*>(&sk[j][c0]);
      const float4 dd = *reinterpret_cast<const float4*>(&sd[j][c0]);
      const float k[4] = {kk.x, kk.y, kk.z, kk.w}, D[4] = {dd.x, dd.y, dd.z, dd.w};
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = sv[j][r0 + i];
      fwd_step(S, k, D, sb[j], v);
    }
  }
}

// ---- pass 2: reverse walk ----
// shared memory per block of tokens: k, q, D, v, dout [kBwdBlock][128] fp32
// each, beta [kBwdBlock], and the per-warp terms of one token's record [warps][kBwdRec]
constexpr int kBwdSmK = 0, kBwdSmQ = kBwdBlock * 128, kBwdSmD = 2 * kBwdBlock * 128;
constexpr int kBwdSmV = 3 * kBwdBlock * 128, kBwdSmO = 4 * kBwdBlock * 128;
constexpr int kBwdSmB = 5 * kBwdBlock * 128, kBwdSmR = kBwdSmB + kBwdBlock;
static_assert(kBwdSmR % 4 == 0 && kBwdRec % 4 == 0, "float4 access to the record rows");
// (with 16 / R warps per CTA, only their record rows are used)
constexpr int kBwdSmem = (kBwdSmR + kBwdWarps * kBwdRec) * 4;
__host__ __device__ constexpr int bwd_smem_bytes(int warps, bool store = false) {
  return (kBwdSmR + warps * kBwdRec + (store ? kBwdBlock * 8 * warps * kHeadDim : 0)) * 4;
}
constexpr int kBwdStoreWarps = 2;  // CTAs up to this many warps keep the block's states
constexpr int kBwdSmemStore = bwd_smem_bytes(kBwdStoreWarps, true);

// kStore (CTAs of at most 2 warps): the states before the block's tokens are
// computed once, going forward from the checkpoint, and kept in shared memory
// after the record rows ([kBwdBlock][8 rows per warp x warps][128] fp32, each
// thread reading back only what it wrote); otherwise each token's state is
// replayed from the checkpoint.  Both give the same bits.
template <int kGate, bool kL2, bool kStore>
__global__ void __launch_bounds__(kBwdThreads) kda_bwd_kernel(BwdParams p, int rsplit) {
  extern __shared__ float sm[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int64_t H = p.H;
  const int64_t unit = blockIdx.x / rsplit;
  const int rb = (int)(blockIdx.x - unit * rsplit);
  const int64_t n = unit / H;
  const int h = (int)(unit - n * H);
  int64_t bos, eos;
  seq_bounds(p, n, bos, eos);
  const int c0 = 4 * lane, r0 = 8 * (warp + nw * rb);
  float* rec = p.rec + (int64_t)rb * p.rows * H * kBwdRec;  // this row block's record parts
  const int64_t sbase = unit * (int64_t)(kHeadDim * kHeadDim);
  const GateC gc = gate_consts(p, h, c0);
  float ds[8][4];  // dL / d(state row) after the current token
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (p.dfinal) {
      const float4 x = *reinterpret_cast<const float4*>(p.dfinal + sbase + (int64_t)(r0 + i) * kHeadDim + c0);
      ds[i][0] = x.x;
      ds[i][1] = x.y;
      ds[i][2] = x.z;
      ds[i][3] = x.w;
    } else {
      ds[i][0] = ds[i][1] = ds[i][2] = ds[i][3] = 0.f;
    }
  }
  const float* ck = p.ckpt + (h * p.nslots + bos / kBwdBlock + n) * (int64_t)(kHeadDim * kHeadDim);
  const int64_t len = eos - bos;
  const int64_t nblk = (len + kBwdBlock - 1) / kBwdBlock;
  for (int64_t blk = nblk - 1; blk >= 0; --blk) {
    const int64_t t_lo = bos + blk * kBwdBlock;
    const int nt = (int)min((int64_t)kBwdBlock, eos - t_lo);
    __syncthreads();  // the previous block's staging is no longer read
    for (int j = warp; j < nt; j += nw) {  // warp w stages tokens w, w + nw, ...
      const int64_t row = (t_lo + j) * H + h;
      float k[4], q[4], D[4], beta;
      token_inputs<kGate, kL2>(p, row, c0, gc, k, q, D, beta);
      float dov[4], vv[4];
      load4(p.v + row * kHeadDim + c0, vv);
      load4(p.dout + row * kHeadDim + c0, dov);
      *reinterpret_cast<float4*>(sm + kBwdSmK + j * 128 + c0) = make_float4(k[0], k[1], k[2], k[3]);
      *reinterpret_cast<float4*>(sm + kBwdSmQ + j * 128 + c0) = make_float4(q[0], q[1], q[2], q[3]);
      *reinterpret_cast<float4*>(sm + kBwdSmD + j * 128 + c0) = make_float4(D[0], D[1], D[2], D[3]);
      *reinterpret_cast<float4*>(sm + kBwdSmV + j * 128 + c0) = make_float4(vv[0], vv[1], vv[2], vv[3]);
      *reinterpret_cast<float4*>(sm + kBwdSmO + j * 128 + c0) = make_float4(dov[0], dov[1], dov[2], dov[3]);
      if (lane == 0) sm[kBwdSmB + j] = beta;
    }
    __syncthreads();
    float S0[8][4];
    {
      const float* src = ck + blk * (int64_t)(kHeadDim * kHeadDim);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(src + (r0 + i) * kHeadDim + c0);
        S0[i][0] = x.x;
        S0[i][1] = x.y;
        S0[i][2] = x.z;
        S0[i][3] = x.w;
      }
    }
    float* sst = sm + kBwdSmR + nw * kBwdRec;  // stored states (kStore)
    if (kStore) {
      for (int j = 0; j < nt; ++j) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(sst + (j * 8 * nw + 8 * warp + i) * kHeadDim + c0) =
              make_float4(S0[i][0], S0[i][1], S0[i][2], S0[i][3]);
        if (j + 1 < nt) {
          float k[4], D[4], v[8];
          const float4 kk = *reinterpret_cast<const float4*>(sm + kBwdSmK + j * 128 + c0);
          const float4 dd = *reinterpret_cast<const float4*>(sm + kBwdSmD + j * 128 + c0);
          k[0] = kk.x; k[1] = kk.y; k[2] = kk.z; k[3] = kk.w;
          D[0] = dd.x; D[1] = dd.y; D[2] = dd.z; D[3] = dd.w;
#pragma unroll
          for (int i = 0; i < 8; ++i) v[i] = sm[kBwdSmV + j * 128 + r0 + i];
          fwd_step(S0, k, D, sm[kBwdSmB + j], v);
        }
      }
    }
    for (int j = nt - 1; j >= 0; --j) {
      // state before token j of the block: stored, or replayed from the checkpoint
      float S[8][4];
      if (kStore) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = *reinterpret_cast<const float4*>(sst + (j * 8 * nw + 8 * warp + i) * kHeadDim + c0);
          S[i][0] = x.x;
          S[i][1] = x.y;
          S[i][2] = x.z;
          S[i][3] = x.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) S[i][c] = S0[i][c];
      }
      for (int jj = 0; jj < (kStore ? 0 : j); ++jj) {
        float k[4], D[4], v[8];
        const float4 kk = *reinterpret_cast<const float4*>(sm + kBwdSmK + jj * 128 + c0);
        const float4 dd = *reinterpret_cast<const float4*>(sm + kBwdSmD + jj * 128 + c0);
        k[0] = kk.x; k[1] = kk.y; k[2] = kk.z; k[3] = kk.w;
        D[0] = dd.x; D[1] = dd.y; D[2] = dd.z; D[3] = dd.w;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = sm[kBwdSmV + jj * 128 + r0 + i];
        fwd_step(S, k, D, sm[kBwdSmB + jj], v);
      }
      // reverse step of token j
      float k[4], q[4], D[4];
      {
        const float4 kk = *reinterpret_cast<const float4*>(sm + kBwdSmK + j * 128 + c0);
        const float4 qq = *reinterpret_cast<const float4*>(sm + kBwdSmQ + j * 128 + c0);
        const float4 dd = *reinterpret_cast<const float4*>(sm + kBwdSmD + j * 128 + c0);
        k[0] = kk.x; k[1] = kk.y; k[2] = kk.z; k[3] = kk.w;
        q[0] = qq.x; q[1] = qq.y; q[2] = qq.z; q[3] = qq.w;
        D[0] = dd.x; D[1] = dd.y; D[2] = dd.z; D[3] = dd.w;
      }
      const float beta = sm[kBwdSmB + j];
      float sp[8][4], pr[8];  // s' = s_prev Diag(D)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        pr[i] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          sp[i][c] = S[i][c] * D[c];
          pr[i] += sp[i][c] * k[c];
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) pr[i] = warp_sum_b(pr[i]);
      float gq[4] = {0.f, 0.f, 0.f, 0.f}, gk[4] = {0.f, 0.f, 0.f, 0.f}, gD[4] = {0.f, 0.f, 0.f, 0.f};
      float gb = 0.f;
      float dsk[8], u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float vi = sm[kBwdSmV + j * 128 + r0 + i], doi = sm[kBwdSmO + j * 128 + r0 + i] * p.scale;
        u[i] = vi - pr[i];
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float snew = sp[i][c] + beta * u[i] * k[c];
          gq[c] += doi * snew;
          ds[i][c] += doi * q[c];
          acc += ds[i][c] * k[c];
        }
        dsk[i] = acc;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) dsk[i] = warp_sum_b(dsk[i]);
      float duv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        gb += u[i] * dsk[i];
        const float du = beta * dsk[i];
        duv[i] = du;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          gk[c] += beta * u[i] * ds[i][c] - du * sp[i][c];
          const float dsp = ds[i][c] - du * k[c];
          gD[c] += dsp * S[i][c];
          ds[i][c] = dsp * D[c];
        }
      }
      const int64_t row = (t_lo + j) * H + h;
      if (lane == 0)
        *reinterpret_cast<float4*>(p.dv + row * kHeadDim + r0) = make_float4(duv[0], duv[1], duv[2], duv[3]);
      else if (lane == 1)
        *reinterpret_cast<float4*>(p.dv + row * kHeadDim + r0 + 4) = make_float4(duv[4], duv[5], duv[6], duv[7]);
      // the token's record: this warp's terms, then the sum over the CTA's warps
      float* rw = sm + kBwdSmR + warp * kBwdRec;
      *reinterpret_cast<float4*>(rw + c0) = make_float4(gq[0], gq[1], gq[2], gq[3]);
      *reinterpret_cast<float4*>(rw + kHeadDim + c0) = make_float4(gk[0], gk[1], gk[2], gk[3]);
      *reinterpret_cast<float4*>(rw + 2 * kHeadDim + c0) = make_float4(gD[0], gD[1], gD[2], gD[3]);
      if (lane == 0) rw[kBwdRecBeta] = gb;
      __syncthreads();
      for (int e = threadIdx.x; e <= kBwdRecBeta; e += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < nw; ++w) s += sm[kBwdSmR + w * kBwdRec + e];
        rec[row * kBwdRec + e] = s;
      }
      __syncthreads();
    }
  }
  if (p.dinit) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      *reinterpret_cast<float4*>(p.dinit + sbase + (int64_t)(r0 + i) * kHeadDim + c0) =
          make_float4(ds[i][0], ds[i][1], ds[i][2], ds[i][3]);
  }
}

// ---- pass 3: finalize ----
// one warp per (run of up to 64 packed token rows, head); lane = 4 channels.
// Works on token rows, not sequences: every row has its record.
constexpr int kFinRun = 64;

template <int kGate, bool kL2>
__global__ void __launch_bounds__(256) kda_bwd_finalize_kernel(BwdParams p, int rsplit) {
  const int lane = threadIdx.x & 31;
  const int64_t H = p.H, rows = p.rows;
  const int64_t runs = (rows + kFinRun - 1) / kFinRun;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (wid >= runs * H) return;
  const int64_t run = wid / H;
  const int h = (int)(wid - run * H);
  const int64_t t0 = run * kFinRun, t1 = min(t0 + kFinRun, rows);
  const int c0 = 4 * lane;
  const GateC gc = gate_consts(p, h, c0);
  float acc_dtb[4] = {0.f, 0.f, 0.f, 0.f}, acc_alog = 0.f;
  for (int64_t t = t0; t < t1; ++t) {
    const int64_t row = t * H + h;
    // the record: its R row-block parts summed in order
    const int64_t part = p.rows * H * kBwdRec;
    float4 gq4 = make_float4(0.f, 0.f, 0.f, 0.f), gk4 = gq4, gD4 = gq4;
    float recb = 0.f;
    for (int r = 0; r < rsplit; ++r) {
      const float* rp = p.rec + r * part + row * kBwdRec;
      const float4 a = *reinterpret_cast<const float4*>(rp + c0);
      const float4 b = *reinterpret_cast<const float4*>(rp + kHeadDim + c0);
      const float4 c = *reinterpret_cast<const float4*>(rp + 2 * kHeadDim + c0);
      gq4 = make_float4(gq4.x + a.x, gq4.y + a.y, gq4.z + a.z, gq4.w + a.w);
      gk4 = make_float4(gk4.x + b.x, gk4.y + b.y, gk4.z + b.z, gk4.w + b.w);
      gD4 = make_float4(gD4.x + c.x, gD4.y + c.y, gD4.z + c.z, gD4.w + c.w);
      if (lane == 0) recb += rp[kBwdRecBeta];
    }
    float q[4], k[4], g[4];
    load4(p.q + row * kHeadDim + c0, q);
    load4(p.k + row * kHeadDim + c0, k);
    if (p.g32) {
      const float4 x = *reinterpret_cast<const float4*>(p.g32 + row * kHeadDim + c0);
      g[0] = x.x; g[1] = x.y; g[2] = x.z; g[3] = x.w;
    } else {
      load4(p.g + row * kHeadDim + c0, g);
    }
    const float gq[4] = {gq4.x, gq4.y, gq4.z, gq4.w}, gk[4] = {gk4.x, gk4.y, gk4.z, gk4.w};
    const float gD[4] = {gD4.x, gD4.y, gD4.z, gD4.w};
    float dq[4], dk[4];
    if (kL2) {  // x_hat = x / r, r = sqrt(|x|^2 + eps): dx = dx_hat / r - x (x . dx_hat) / r^3
      const float nq = warp_sum_b(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]) + 1e-6f;
      const float nk = warp_sum_b(k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3]) + 1e-6f;
      const float xq = warp_sum_b(q[0] * gq[0] + q[1] * gq[1] + q[2] * gq[2] + q[3] * gq[3]);
      const float xk = warp_sum_b(k[0] * gk[0] + k[1] * gk[1] + k[2] * gk[2] + k[3] * gk[3]);
      const float rq = rsqrtf(nq), rk = rsqrtf(nk);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        dq[c] = gq[c] * rq - q[c] * xq * rq * rq * rq;
        dk[c] = gk[c] * rk - k[c] * xk * rk * rk * rk;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        dq[c] = gq[c];
        dk[c] = gk[c];
      }
    }
    // gate: dL/da = dL/dD * D; a = f(z), z = g + dt_bias
    float dg[4], dal = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float z = kGate == kGateLogspace ? g[c] : g[c] + gc.dtb[c];
      if (kGate == kGateLogspace) {
        dg[c] = gD[c] * expf(z);
      } else if (kGate == kGateUnsafe) {
        const float sp = fmaxf(z, 0.f) + log1pf(expf(-fabsf(z)));  // softplus
        const float a = -gc.amul * sp;
        const float da = gD[c] * expf(a);
        const float sig = 1.0f / (1.0f + expf(-z));
        dg[c] = -gc.amul * sig * da;
        dal += da * a;                                              // da/dA_log = a
      } else {
        const float x = gc.amul * z;
        const float sig = 1.0f / (1.0f + expf(-x));
        const float a = gc.lb * sig;
        const float da = gD[c] * expf(a);
        const float dsig = sig * (1.0f - sig);
        dg[c] = gc.lb * gc.amul * dsig * da;
        dal += da * gc.lb * dsig * x;                                // da/dA_log = lb sig' amul z
      }
      acc_dtb[c] += dg[c];
    }
    acc_alog += warp_sum_b(dal);
    *reinterpret_cast<float4*>(p.dq + row * kHeadDim + c0) = make_float4(dq[0], dq[1], dq[2], dq[3]);
    *reinterpret_cast<float4*>(p.dk + row * kHeadDim + c0) = make_float4(dk[0], dk[1], dk[2], dk[3]);
    *reinterpret_cast<float4*>(p.dg + row * kHeadDim + c0) = make_float4(dg[0], dg[1], dg[2], dg[3]);
    if (lane == 0) {
      const float braw = bf16_to_f(p.beta[row]);
      float db = recb;
      if (!p.beta_prob) {
        const float bt = 1.0f / (1.0f + expf(-braw));
        db *= bt * (1.0f - bt);
      }
      p.dbeta[row] = db;
    }
  }
  if (kGate != kGateLogspace) {
    if (p.ddt_bias)
      for (int c = 0; c < 4; ++c) atomicAdd(p.ddt_bias + h * kHeadDim + c0 + c, acc_dtb[c]);
    if (p.dA_log && p.A_log && lane == 0) atomicAdd(p.dA_log + h, acc_alog);
  }
}

template <int kGate, bool kL2>
static void launch_bwd_variant(const BwdParams& p, int rsplit, cudaStream_t s, void* const* ev) {
  auto mark = [&](int i) {
    if (ev && ev[i]) cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev[i]), s);
  };
  const unsigned ctas = (unsigned)(p.N * p.H * rsplit);
  const int warps_per_cta = kBwdWarps / rsplit;
  kda_bwd_ckpt_kernel<kGate, kL2><<<ctas, 32 * warps_per_cta, 0, s>>>(p, rsplit);
  mark(1);
  if (warps_per_cta <= kBwdStoreWarps)
    kda_bwd_kernel<kGate, kL2, true><<<ctas, 32 * warps_per_cta, bwd_smem_bytes(warps_per_cta, true), s>>>(p, rsplit);
  else
    kda_bwd_kernel<kGate, kL2, false><<<ctas, 32 * warps_per_cta, bwd_smem_bytes(warps_per_cta), s>>>(p, rsplit);
  mark(2);
  const int64_t warps = (p.rows + kFinRun - 1) / kFinRun * p.H;
  if (warps > 0) kda_bwd_finalize_kernel<kGate, kL2><<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(p, rsplit);
  mark(3);
}

// ev: optional events (cudaEvent_t, each may be null) recorded after the
// checkpoint, reverse and finalize launches (entries 1, 2, 3).
static void launch_bwd_events(const BwdParams& p, int rsplit, cudaStream_t s, void* const* ev) {
  if (p.N * p.H == 0) return;
  const bool l2 = p.l2norm != 0;
  switch (p.gate_mode) {
    case kGateUnsafe:
      if (l2) launch_bwd_variant<kGateUnsafe, true>(p, rsplit, s, ev);
      else launch_bwd_variant<kGateUnsafe, false>(p, rsplit, s, ev);
      break;
    case kGateLogspace:
      if (l2) launch_bwd_variant<kGateLogspace, true>(p, rsplit, s, ev);
      else launch_bwd_variant<kGateLogspace, false>(p, rsplit, s, ev);
      break;
    default:
      if (l2) launch_bwd_variant<kGateSafe, true>(p, rsplit, s, ev);
      else launch_bwd_variant<kGateSafe, false>(p, rsplit, s, ev);
  }
}

// Row blocks per (sequence, head): the largest power of two up to 16 that keeps
// the CTAs of a launch within two per SM (1 when the units alone fill the GPU,
// and on the host without a device).
static int bwd_row_split(int64_t units) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  int r = 1;
  while (r < kBwdWarps && units * (2 * r) <= 2 * (int64_t)sms) r *= 2;
  return r;
}

void launch_bwd(const BwdParams& p, cudaStream_t s) { launch_bwd_events(p, bwd_row_split(p.N * p.H), s, nullptr); }

cudaError_t prepare_bwd() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  const void* fns[] = {(const void*)kda_bwd_kernel<kGateSafe, true, false>,
                       (const void*)kda_bwd_kernel<kGateSafe, false, false>,
                       (const void*)kda_bwd_kernel<kGateUnsafe, true, false>,
                       (const void*)kda_bwd_kernel<kGateUnsafe, false, false>,
                       (const void*)kda_bwd_kernel<kGateLogspace, true, false>,
                       (const void*)kda_bwd_kernel<kGateLogspace, false, false>};
  const void* fns_store[] = {(const void*)kda_bwd_kernel<kGateSafe, true, true>,
                             (const void*)kda_bwd_kernel<kGateSafe, false, true>,
                             (const void*)kda_bwd_kernel<kGateUnsafe, true, true>,
                             (const void*)kda_bwd_kernel<kGateUnsafe, false, true>,
                             (const void*)kda_bwd_kernel<kGateLogspace, true, true>,
                             (const void*)kda_bwd_kernel<kGateLogspace, false, true>};
  for (const void* f : fns) {
    const cudaError_t e = cudaFuncSetAttribute(f, attr, kBwdSmem);
    if (e != cudaSuccess) return e;
  }
  for (const void* f : fns_store) {
    const cudaError_t e = cudaFuncSetAttribute(f, attr, kBwdSmemStore);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Checkpoint slots per head: sequence n (rows bos .. eos) uses slots
// bos / kBwdBlock + n + b for its blocks b, which never collide:
// rows / kBwdBlock + N + 1 cover them all.
int64_t bwd_slots(int64_t rows, int64_t N) { return rows / kBwdBlock + N + 1; }
int bwd_record_floats() { return kBwdRec; }

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
  const int64_t rows = a->fwd.B * a->fwd.T, H = a->fwd.H, N = a->fwd.N;
  const size_t ckpt = (size_t)H * (size_t)bwd_slots(rows, N) * kHeadDim * kHeadDim * sizeof(float);
  const size_t rec = (size_t)rows * (size_t)H * (size_t)bwd_record_floats() * sizeof(float) *
                     (size_t)bwd_row_split(N * H);
  return round256(ckpt) + round256(rec);
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
  const size_t ckpt_bytes = round256((size_t)H * (size_t)bwd_slots(rows, f.N) * kHeadDim * kHeadDim * sizeof(float));
  const int rsplit = bwd_row_split(f.N * H);
  const size_t rec_bytes =
      (size_t)rows * (size_t)H * (size_t)bwd_record_floats() * sizeof(float) * (size_t)rsplit;
  const uint32_t gate = f.flags & (KDA_GATE_SAFE | KDA_GATE_UNSAFE | KDA_GATE_LOGSPACE);
  bool ok = true;
  auto chk = [&](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // sums over tokens accumulate from zero; with packed sequences, rows of a
  // sequence skipped for bad bounds keep zero gradients
  if (a->dA_log && gate != KDA_GATE_LOGSPACE) chk(cudaMemsetAsync(a->dA_log, 0, H * sizeof(float), s));
  if (a->ddt_bias && gate != KDA_GATE_LOGSPACE)
    chk(cudaMemsetAsync(a->ddt_bias, 0, H * kHeadDim * sizeof(float), s));
  if (f.cu_seqlens && rows > 0) {
    chk(cudaMemsetAsync(a->dv, 0, (size_t)rows * H * kHeadDim * sizeof(float), s));
    chk(cudaMemsetAsync(ws + ckpt_bytes, 0, rec_bytes, s));
  }
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
  p.N = f.N;
  p.T = f.T;
  p.H = H;
  p.rows = rows;
  p.nslots = bwd_slots(rows, f.N);
  p.status = f.cu_seqlens ? status : nullptr;
  p.ckpt = reinterpret_cast<float*>(ws);
  p.rec = reinterpret_cast<float*>(ws + ckpt_bytes);
  p.dq = a->dq;
  p.dk = a->dk;
  p.dv = a->dv;
  p.dg = a->dg;
  p.dbeta = a->dbeta;
  p.dA_log = gate != KDA_GATE_LOGSPACE ? a->dA_log : nullptr;
  p.ddt_bias = gate != KDA_GATE_LOGSPACE ? a->ddt_bias : nullptr;
  p.dinit = a->dinitial_state;
  launch_bwd_events(p, rsplit, s, events);
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
