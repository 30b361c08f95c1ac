// Intra-chunk stage of the KDA forward pass: one CTA per (64-token chunk, head).
//
// Computes, for its chunk, everything that does not depend on the recurrent
// state and stores it in the workspace slot of (chunk, head):
//   * the gate activation and the in-chunk cumulative decay (the "gate.py"
//     stage of the fla-kda code map: gate activation + cumulative decay),
//   * optional q/k L2 normalisation,
//   * A (beta-scaled strictly-lower decayed K K^T) and P (lower decayed Q K^T)
//     from 16-token sub-chunks: off-diagonal sub-blocks use paired decay
//     factors whose exponents are both <= 0, diagonal sub-blocks use an
//     offset at the sub-chunk midpoint (fla-kda SKILL.md, "Numerical
//     invariants"; fla-kda skill page on the midpoint offset),
//   * T = (I + A)^-1 Diag(beta) by 16x16 diagonal inverses and block merges
//     (the "solve_tril" / triangular block merge stage),
//   * W = T (K * gamma) and U = T V (the "wy_fast" WY recompute),
//   * q * gamma, k * gamma_C / gamma and gamma_C for the state stage.
//
// Decay factors inside a sub-chunk come from running products of
// d_t = exp(a_t), so every exponent is taken once per (token, channel).
// The A and P operands are stored relative to the cumulative decay at the
// sub-chunk midpoint (after its 8th token); off-diagonal sub-blocks multiply
// in per-channel factors (midpoint -> sub-chunk end -> ... -> next midpoint),
// all <= 1.  For these operands d_t is clamped below at exp(-10), so that the
// midpoint-relative values stay within [e^-80, e^80] for any gate; with the
// safe gate (a_t >= -5) the clamp never acts.  Where it acts, the true pair
// factor and the clamped one are both below exp(-10).  The recurrent-state
// quantities (q gamma, K gamma, k gamma_C / gamma, gamma_C) use the exact d_t.
//
// Precision: the A / P operands are bf16 (they need its exponent range); the
// solve is fp32; T, K gamma, V, W, U and everything written to the workspace
// are fp16 (11-bit significand) with fp32 accumulation.
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

// exp(-10): floor of the per-token decay inside the diagonal-block factors.
constexpr float kDiagDecayFloor = 4.5399929762484854e-05f;

// shared-memory map (bytes)
constexpr int kCsQ = 0;          // tile128: raw q, then bf16 q_hat * xr
constexpr int kCsK = 16384;      // tile128: raw k, then bf16 k_hat * xr
constexpr int kCsKy = 32768;     // tile128: bf16 k_hat * yr
constexpr int kCsKg = 49152;     // tile128: raw g, then fp16 k_hat * gamma
constexpr int kCsV = 65536;      // tile128: v, converted in place to fp16
constexpr int kCsA = 81920;      // fp32 [64][64]: A (lower blocks)
constexpr int kCsInv = 98304;    // fp32 [64][64]: (I + A)^-1 (lower blocks)
constexpr int kCsT = 114688;     // tile64: T = (I + A)^-1 Diag(beta), fp16
constexpr int kCsM = 122880;     // fp32 [3][16][16]: solve scratch
constexpr int kCsD = 125952;     // fp32 [4][128]: exact sub-chunk decay products
constexpr int kCsXm = 128000;    // fp32 [4][128]: clamped product over tokens 0..7 of a sub-chunk
constexpr int kCsYm = 130048;    // fp32 [4][128]: clamped product over tokens 8..15
constexpr int kCsBeta = 134144;  // fp32 [64]
constexpr int kCsRq = 134400;    // fp32 [64]: 1 / |q| (or 1)
constexpr int kCsRk = 134656;    // fp32 [64]: 1 / |k| (or 1)
constexpr int kChunkSmem = 134912;

__device__ __forceinline__ float sigmoidf_fast(float x) {
  return __frcp_rn(1.0f + ex2(-x * kLog2e));
}

// log(1 + e) for e in [0, 1]; a short series where lg2(1 + e) would lose e.
__device__ __forceinline__ float log1p_small(float e) {
  if (e < 0.0078125f) return e * (1.0f - e * (0.5f - e * (1.0f / 3.0f)));
  return lg2(1.0f + e) * 0.69314718055994531f;
}

__device__ __forceinline__ float ld_tile128(const unsigned char* base, int row, int col) {
  return bf16_to_f(*reinterpret_cast<const uint16_t*>(base + swz128(row, col)));
}
__device__ __forceinline__ void st_tile128(unsigned char* base, int row, int col, float x) {
  *reinterpret_cast<__nv_bfloat16*>(base + swz128(row, col)) = __float2bfloat16_rn(x);
}
__device__ __forceinline__ void st_tile128_f16(unsigned char* base, int row, int col, float x) {
  *reinterpret_cast<__half*>(base + swz128(row, col)) = __float2half_rn(x);
}

// Scale the 8 bf16 values of an A fragment (columns ch, ch+1, ch+8, ch+9) by
// per-column factors f[0..3].
__device__ __forceinline__ void scale_afrag(uint32_t (&a)[4], const float (&f)[4]) {
  float2 v;
  v = unpack_bf16(a[0]); a[0] = pack_bf16(v.x * f[0], v.y * f[1]);
  v = unpack_bf16(a[1]); a[1] = pack_bf16(v.x * f[0], v.y * f[1]);
  v = unpack_bf16(a[2]); a[2] = pack_bf16(v.x * f[2], v.y * f[3]);
  v = unpack_bf16(a[3]); a[3] = pack_bf16(v.x * f[2], v.y * f[3]);
}
// Scale a B fragment pair (rows k = ch, ch+1 | ch+8, ch+9) by f[0..3].
__device__ __forceinline__ void scale_bfrag(uint32_t& b0, uint32_t& b1, const float (&f)[4]) {
  float2 v;
  v = unpack_bf16(b0); b0 = pack_bf16(v.x * f[0], v.y * f[1]);
  v = unpack_bf16(b1); b1 = pack_bf16(v.x * f[2], v.y * f[3]);
}

__global__ void __launch_bounds__(256, 1) kda_chunk_kernel(ChunkParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t slot = blockIdx.x;
  const int h = blockIdx.y;
  const int64_t H = p.H;

  // ---- locate the chunk: sequence n, chunk i, first token t0, length L ----
  int64_t n, i, bos, seqlen;
  if (p.cu) {
    if (slot >= p.chunk_off[p.N]) return;
    int64_t lo = 0, hi = p.N - 1;  // largest n with chunk_off[n] <= slot
    while (lo < hi) {
      int64_t mid = (lo + hi + 1) >> 1;
      if (p.chunk_off[mid] <= slot) lo = mid; else hi = mid - 1;
    }
    n = lo;
    i = slot - p.chunk_off[n];
    bos = p.cu[n];
    seqlen = p.cu[n + 1] - bos;
  } else {
    n = slot / p.NT;
    i = slot - n * p.NT;
    bos = n * p.T;
    seqlen = p.T;
  }
  const int64_t t0 = bos + i * kChunk;
  const int L = (int)min((int64_t)kChunk, seqlen - i * kChunk);
  unsigned char* ws = p.ws + (slot * H + h) * (int64_t)kSlotBytes;

  // ---- stage q, k, g, v into swizzled tiles (rows >= L zero-filled) ----
  {
    const uint16_t* src[4] = {p.q, p.k, p.g, p.v};
    const int dstoff[4] = {kCsQ, kCsK, kCsKg, kCsV};
    const uint32_t sbase = smem_u32(smem);
    for (int idx = tid; idx < 4 * 1024; idx += 256) {
      int tsr = idx >> 10, row = (idx >> 4) & 63, ch = idx & 15;
      bool ok = row < L;
      const uint16_t* s = ok ? src[tsr] + ((t0 + row) * H + h) * kHeadDim + ch * 8 : src[tsr];
      cp_async16(sbase + dstoff[tsr] + row * 256 + (((ch ^ (row & 7))) << 4), s, ok ? 16 : 0);
    }
    cp_async_commit();
  }
  float* sBeta = reinterpret_cast<float*>(smem + kCsBeta);
  if (tid < kChunk)
    sBeta[tid] = tid < L ? sigmoidf_fast(bf16_to_f(p.beta[(t0 + tid) * H + h])) : 0.0f;
  cp_async_wait<0>();
  __syncthreads();

  // ---- per-token inverse norms of q and k (warp per token) ----
  float* sRq = reinterpret_cast<float*>(smem + kCsRq);
  float* sRk = reinterpret_cast<float*>(smem + kCsRk);
  for (int t = warp; t < kChunk; t += 8) {
    float rq = 1.0f, rk = 1.0f;
    if (p.l2norm) {
      float sq = 0.f, sk = 0.f;
      int c = lane * 4;
      uint32_t off = swz128(t, c);
      uint2 qv = *reinterpret_cast<const uint2*>(smem + kCsQ + off);
      uint2 kv = *reinterpret_cast<const uint2*>(smem + kCsK + off);
      float2 a0 = unpack_bf16(qv.x), a1 = unpack_bf16(qv.y);
      float2 b0 = unpack_bf16(kv.x), b1 = unpack_bf16(kv.y);
      sq = a0.x * a0.x + a0.y * a0.y + a1.x * a1.x + a1.y * a1.y;
      sk = b0.x * b0.x + b0.y * b0.y + b1.x * b1.x + b1.y * b1.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
      }
      rq = rsqrtf(sq + 1e-6f);
      rk = rsqrtf(sk + 1e-6f);
    }
    if (lane == 0) { sRq[t] = rq; sRk[t] = rk; }
  }

  // ---- gate activation and per-sub-chunk decay products ----
  // thread -> channel c, sub-chunks rb0 and rb0 + 2
  const int c = tid & 127;
  const int rb0 = tid >> 7;
  float d[2][kSub];
  float* sD = reinterpret_cast<float*>(smem + kCsD);
  float* sXm = reinterpret_cast<float*>(smem + kCsXm);
  float* sYm = reinterpret_cast<float*>(smem + kCsYm);
  {
    const float dtb = p.dt_bias ? p.dt_bias[h * kHeadDim + c] : 0.0f;
    const float amul = p.A_log ? expf(p.A_log[h]) : 1.0f;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int rb = rb0 + 2 * b;
      float D = 1.f, xm = 1.f, ym = 1.f;
#pragma unroll
      for (int j = 0; j < kSub; ++j) {
        const int t = rb * kSub + j;
        const float z = ld_tile128(smem + kCsKg, t, c) + dtb;
        float a;
        if (p.gate_unsafe) {
          float e = ex2(-fabsf(z) * kLog2e);
          a = -amul * (fmaxf(z, 0.0f) + log1p_small(e));
        } else {
          a = p.lower_bound * sigmoidf_fast(amul * z);
        }
        float dj = t < L ? ex2(a * kLog2e) : 1.0f;
        d[b][j] = dj;
        D *= dj;
        if (j < 8) xm *= fmaxf(dj, kDiagDecayFloor); else ym *= fmaxf(dj, kDiagDecayFloor);
      }
      sD[rb * 128 + c] = D;
      sXm[rb * 128 + c] = xm;
      sYm[rb * 128 + c] = ym;
    }
  }
  __syncthreads();

  // ---- operands ----
  //  exact, chunk relative:   gamma_j = prod_{s<=j} d_s   -> K gamma (smem), q gamma (ws)
  //  exact, chunk-end rel.:   gamma_C / gamma_j            -> k_hat (ws)
  //  clamped, midpoint rel.:  xr_j = e^{lam_j - lam_7}, yr_j = 1 / xr_j  -> A / P operands
  {
    __half* gQg = reinterpret_cast<__half*>(ws + kSlotQg);
    __half* gKh = reinterpret_cast<__half*>(ws + kSlotKh);
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int rb = rb0 + 2 * b;
      float pre = 1.f, suf = 1.f;
      for (int s = 0; s < 4; ++s) {
        float Ds = sD[s * 128 + c];
        if (s < rb) pre *= Ds;
        if (s > rb) suf *= Ds;
      }
      float xe[kSub], ye[kSub], mr[kSub];
      {
        float x = pre;
#pragma unroll
        for (int jj = 0; jj < kSub; ++jj) { x *= d[b][jj]; xe[jj] = x; }
        float y = suf;
#pragma unroll
        for (int jj = kSub - 1; jj >= 0; --jj) { ye[jj] = y; y *= d[b][jj]; }
        // mr_j = prod_{s=j+1..7} dc_s for j <= 7, prod_{s=8..j} dc_s for j >= 8
        float m = 1.f;
#pragma unroll
        for (int jj = 7; jj >= 0; --jj) { mr[jj] = m; m *= fmaxf(d[b][jj], kDiagDecayFloor); }
        m = 1.f;
#pragma unroll
        for (int jj = 8; jj < kSub; ++jj) { m *= fmaxf(d[b][jj], kDiagDecayFloor); mr[jj] = m; }
      }
#pragma unroll
      for (int jj = 0; jj < kSub; ++jj) {
        const int t = rb * kSub + jj;
        const float kh = ld_tile128(smem + kCsK, t, c) * sRk[t];
        const float qh = ld_tile128(smem + kCsQ, t, c) * sRq[t];
        const float inv = __frcp_rn(mr[jj]);
        const float xr = jj < 8 ? inv : mr[jj];
        const float yr = jj < 8 ? mr[jj] : inv;
        st_tile128(smem + kCsK, t, c, kh * xr);
        st_tile128(smem + kCsQ, t, c, qh * xr);
        st_tile128(smem + kCsKy, t, c, kh * yr);
        st_tile128_f16(smem + kCsKg, t, c, kh * xe[jj]);
        st_tile128_f16(smem + kCsV, t, c, ld_tile128(smem + kCsV, t, c));
        gQg[t * kHeadDim + c] = __float2half_rn(qh * xe[jj]);
        gKh[t * kHeadDim + c] = __float2half_rn(kh * ye[jj]);
      }
    }
    if (rb0 == 0) {
      float gc = sD[c] * sD[128 + c] * sD[256 + c] * sD[384 + c];
      reinterpret_cast<float*>(ws + kSlotGc)[c] = gc;
    }
  }
  __syncthreads();

  const uint32_t sbase = smem_u32(smem);
  const int g = lane >> 2, q4 = lane & 3;
  float* sA = reinterpret_cast<float*>(smem + kCsA);
  float* sInv = reinterpret_cast<float*>(smem + kCsInv);

  // ---- A (warps 0-3) and P (warps 4-7): row sub-block r, column sub-blocks c <= r ----
  // Diagonal sub-blocks: the midpoint-relative operands multiply directly.
  // Off-diagonal (cb < r): the left operands get the per-channel factor
  //   xm[r] * prod_{cb<s<r} xm[s] ym[s]   (-> relative to the end of sub-chunk cb)
  // and the right operands ym[cb] (-> relative to the end of sub-chunk cb), so
  // each side is <= |k| and underflows only where the pair factor itself does.
  {
    const int mat = warp >> 2, r = warp & 3;
    __half* gP = reinterpret_cast<__half*>(ws + kSlotP);
    for (int cb = 0; cb < 4; ++cb) {
      float acc[2][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
      const bool active = cb <= r;
      if (active) {
#pragma unroll 2
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t a[4];
          lda_128(a, sbase + (mat ? kCsQ : kCsK), 16 * r, 16 * kk, lane);
          uint32_t b[4];
          ldb_nk_128(b, sbase + kCsKy, 16 * cb, 16 * kk, lane);
          if (cb < r) {
            const int ch = 16 * kk + 2 * q4;
            const int chs[4] = {ch, ch + 1, ch + 8, ch + 9};
            float fa[4], fb[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float e = sXm[r * 128 + chs[u]];
              for (int s = cb + 1; s < r; ++s) e *= sXm[s * 128 + chs[u]] * sYm[s * 128 + chs[u]];
              fa[u] = e;
              fb[u] = sYm[cb * 128 + chs[u]];
            }
            scale_afrag(a, fa);
            scale_bfrag(b[0], b[1], fb);
            scale_bfrag(b[2], b[3], fb);
          }
          mma_bf16(acc[0], a, b[0], b[1]);
          mma_bf16(acc[1], a, b[2], b[3]);
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int row = 16 * r + g + 8 * hf;
          const int col = 16 * cb + 8 * nt + 2 * q4;
          float v0 = acc[nt][2 * hf], v1 = acc[nt][2 * hf + 1];
          if (mat == 0) {
            const bool k0 = active && (cb < r || col < row);
            const bool k1 = active && (cb < r || col + 1 < row);
            const float bt = sBeta[row];
            sA[row * 64 + col] = k0 ? v0 * bt : 0.f;
            sA[row * 64 + col + 1] = k1 ? v1 * bt : 0.f;
          } else {
            const bool k0 = active && (cb < r || col <= row);
            const bool k1 = active && (cb < r || col + 1 <= row);
            *reinterpret_cast<uint32_t*>(gP + row * 64 + col) =
                pack_f16(k0 ? v0 : 0.f, k1 ? v1 : 0.f);
          }
        }
      }
    }
  }
  __syncthreads();

  // ---- solve: inverses of the four 16x16 unit-lower diagonal blocks ----
  if (warp < 4 && lane < 16) {
    const int j = lane, o = 16 * warp;
    float x[kSub];
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii) {
      float acc = 0.f;
#pragma unroll
      for (int s = 0; s < ii; ++s) acc += sA[(o + ii) * 64 + o + s] * x[s];
      x[ii] = (ii == j) ? 1.f : (ii < j ? 0.f : -acc);
    }
#pragma unroll
    for (int ii = 0; ii < kSub; ++ii) sInv[(o + ii) * 64 + o + j] = x[ii];
  }
  __syncthreads();
  // ---- block merges: Inv_rc = -X_r * sum_{s=c}^{r-1} A_rs Inv_sc, by distance r-c ----
  {
    float* sM = reinterpret_cast<float*>(smem + kCsM);
    for (int dist = 1; dist < 4; ++dist) {
      const int cnt = 4 - dist;
      for (int idx = tid; idx < cnt * 256; idx += 256) {
        const int tile = idx >> 8, e = idx & 255, ii = e >> 4, jj = e & 15;
        const int r = dist + tile, cb = r - dist;
        float acc = 0.f;
        for (int s = cb; s < r; ++s)
#pragma unroll
          for (int u = 0; u < 16; ++u)
            acc += sA[(16 * r + ii) * 64 + 16 * s + u] * sInv[(16 * s + u) * 64 + 16 * cb + jj];
        sM[tile * 256 + e] = acc;
      }
      __syncthreads();
      for (int idx = tid; idx < cnt * 256; idx += 256) {
        const int tile = idx >> 8, e = idx & 255, ii = e >> 4, jj = e & 15;
        const int r = dist + tile, cb = r - dist;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u)
          acc += sInv[(16 * r + ii) * 64 + 16 * r + u] * sM[tile * 256 + u * 16 + jj];
        sInv[(16 * r + ii) * 64 + 16 * cb + jj] = -acc;
      }
      __syncthreads();
    }
  }
  // ---- T = Inv Diag(beta) as an fp16 operand ----
  for (int idx = tid; idx < 64 * 64; idx += 256) {
    const int ii = idx >> 6, jj = idx & 63;
    const float val = jj <= ii ? sInv[ii * 64 + jj] * sBeta[jj] : 0.f;
    *reinterpret_cast<__half*>(smem + kCsT + swz64(ii, jj)) = __float2half_rn(val);
  }
  __syncthreads();

  // ---- W = T (K gamma) (warps 0-3) and U = T V (warps 4-7), row sub-block r, fp16 ----
  {
    const int mat = warp >> 2, r = warp & 3;
    float acc[16][4];
#pragma unroll
    for (int a = 0; a < 16; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
    for (int cb = 0; cb <= r; ++cb) {
      uint32_t a[4];
      lda_64(a, sbase + kCsT, 16 * r, 16 * cb, lane);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b[4];
        ldb_kn_128(b, sbase + (mat ? kCsV : kCsKg), 16 * np, 16 * cb, lane);
        mma_f16(acc[2 * np], a, b[0], b[1]);
        mma_f16(acc[2 * np + 1], a, b[2], b[3]);
      }
    }
    __half* out = reinterpret_cast<__half*>(ws + (mat ? kSlotU : kSlotW));
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const int row = 16 * r + g, col = 8 * nt + 2 * q4;
      *reinterpret_cast<uint32_t*>(out + row * kHeadDim + col) = pack_f16(acc[nt][0], acc[nt][1]);
      *reinterpret_cast<uint32_t*>(out + (row + 8) * kHeadDim + col) =
          pack_f16(acc[nt][2], acc[nt][3]);
    }
  }
}

void launch_chunk_kernel(const ChunkParams& p, int64_t num_slots, cudaStream_t stream) {
  kda_chunk_kernel<<<dim3((unsigned)num_slots, (unsigned)p.H), 256, kChunkSmem, stream>>>(p);
}

cudaError_t prepare_chunk_kernel() {
  return cudaFuncSetAttribute(kda_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kChunkSmem);
}

}  // namespace kda
