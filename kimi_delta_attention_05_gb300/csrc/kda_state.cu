// Recurrent stage of the KDA forward pass: one CTA per (sequence, head,
// 64-wide value tile), walking the chunks of its sequence in order.
//
// Per chunk, with S the state (rows = value index, columns = key index) at
// the chunk start and the intra-chunk quantities of the workspace slot:
//   U_new = U - W S^T                     (delta-rule correction, WY form)
//   O     = scale (Q_gamma S^T + P U_new)  (inter + intra read-out, fused as in
//                                          the chunk_o stage of the fla code map)
//   S     = S Diag(gamma_C) + U_new^T K_hat   (chunk_delta_h state update)
// Each warp owns 16 value rows of S in mma accumulator registers (fp32); the
// accumulator layout is reused directly as the fp16 left operand of the next
// product, so the sequential chain never leaves the register file.  All
// operands are fp16 (11-bit significand) with fp32 accumulation; the state
// itself stays fp32.
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

constexpr int kStW = 0;
constexpr int kStQg = 16384;
constexpr int kStKh = 32768;
constexpr int kStP = 49152;     // tile64 [t][s]
constexpr int kStU = 57344;     // tile64 [t][v_local]
constexpr int kStGc = 65536;    // fp32 [128]
constexpr int kStBuf = 66048;   // one chunk's operands
constexpr int kStO = 2 * kStBuf;  // tile64 [t][v_local] output staging
constexpr int kStateSmem = kStO + 8192;
constexpr int kVTile = 64;

__device__ __forceinline__ void load_chunk_operands(unsigned char* buf, const unsigned char* src,
                                                    int v0, int tid) {
  const uint32_t dbase = smem_u32(buf);
  for (int idx = tid; idx < 4128; idx += 128) {
    uint32_t dst;
    const unsigned char* s;
    if (idx < 3072) {
      const int m = idx >> 10, row = (idx >> 4) & 63, ch = idx & 15;
      const int soff = m == 0 ? kSlotW : (m == 1 ? kSlotQg : kSlotKh);
      dst = dbase + m * 16384 + row * 256 + ((ch ^ (row & 7)) << 4);
      s = src + soff + row * 256 + ch * 16;
    } else if (idx < 3584) {
      const int e = idx - 3072, row = e >> 3, ch = e & 7;
      dst = dbase + kStP + row * 128 + ((ch ^ (row & 7)) << 4);
      s = src + kSlotP + row * 128 + ch * 16;
    } else if (idx < 4096) {
      const int e = idx - 3584, row = e >> 3, ch = e & 7;
      dst = dbase + kStU + row * 128 + ((ch ^ (row & 7)) << 4);
      s = src + kSlotU + row * 256 + ((v0 >> 3) + ch) * 16;
    } else {
      const int e = idx - 4096;
      dst = dbase + kStGc + e * 16;
      s = src + kSlotGc + e * 16;
    }
    cp_async16(dst, s, 16);
  }
}

__global__ void __launch_bounds__(128, 1) kda_state_kernel(StateParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int64_t H = p.H;
  const int64_t unit = blockIdx.x >> 1;
  const int v0 = (blockIdx.x & 1) * kVTile;
  const int64_t n = unit / H;
  const int h = (int)(unit - n * H);

  int64_t bos, len, slot0;
  if (p.cu) {
    bos = p.cu[n];
    len = p.cu[n + 1] - bos;
    slot0 = p.chunk_off[n];
  } else {
    bos = n * p.T;
    len = p.T;
    slot0 = n * p.NT;
  }
  const int64_t nch = (len + kChunk - 1) / kChunk;

  // ---- initial state into accumulator fragments ----
  float s[16][4];
  const int vr0 = v0 + 16 * warp + g;  // value rows vr0 and vr0 + 8
  {
    const int64_t sbase = (n * H + h) * (int64_t)(kHeadDim * kHeadDim);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = 8 * j + 2 * q4;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        float x0 = 0.f, x1 = 0.f;
        if (p.init) {
          const int64_t off = sbase + (int64_t)(vr0 + 8 * hf) * kHeadDim + col;
          if (p.state_bf16) {
            float2 f = unpack_bf16(*reinterpret_cast<const uint32_t*>(
                reinterpret_cast<const uint16_t*>(p.init) + off));
            x0 = f.x; x1 = f.y;
          } else {
            float2 f = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(p.init) + off);
            x0 = f.x; x1 = f.y;
          }
        }
        s[j][2 * hf] = x0;
        s[j][2 * hf + 1] = x1;
      }
    }
  }

  const unsigned char* ws = p.ws;
  auto slot_ptr = [&](int64_t ci) {
    return ws + ((slot0 + ci) * H + h) * (int64_t)kSlotBytes;
  };
  if (nch > 0) load_chunk_operands(smem, slot_ptr(0), v0, tid);
  cp_async_commit();
  if (nch > 1) load_chunk_operands(smem + kStBuf, slot_ptr(1), v0, tid);
  cp_async_commit();

  const uint32_t sb = smem_u32(smem);
  for (int64_t ci = 0; ci < nch; ++ci) {
    const int cur = (int)(ci & 1);
    const uint32_t bufa = sb + cur * kStBuf;
    const unsigned char* buf = smem + cur * kStBuf;
    cp_async_wait<1>();
    __syncthreads();

    // state -> fp16 left operand over the key dimension (8 k16 steps)
    uint32_t sa[8][4];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      sa[kk][0] = pack_f16(s[2 * kk][0], s[2 * kk][1]);
      sa[kk][1] = pack_f16(s[2 * kk][2], s[2 * kk][3]);
      sa[kk][2] = pack_f16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      sa[kk][3] = pack_f16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
    }

    // X = S W^T  [16 v x 64 t];  U_new^T = U^T - X
    float un[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) un[a][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldb_nk_128(b, bufa + kStW, 16 * np, 16 * kk, lane);
        mma_f16(un[2 * np], sa[kk], b[0], b[1]);
        mma_f16(un[2 * np + 1], sa[kk], b[2], b[3]);
      }
    }
    const int vl = 16 * warp + g;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = 8 * j + 2 * q4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tt = t + (e & 1), vv = vl + 8 * (e >> 1);
        const float u = f16_to_f(*reinterpret_cast<const uint16_t*>(buf + kStU + swz64(tt, vv)));
        un[j][e] = u - un[j][e];
      }
    }
    uint32_t ua[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      ua[kk][0] = pack_f16(un[2 * kk][0], un[2 * kk][1]);
      ua[kk][1] = pack_f16(un[2 * kk][2], un[2 * kk][3]);
      ua[kk][2] = pack_f16(un[2 * kk + 1][0], un[2 * kk + 1][1]);
      ua[kk][3] = pack_f16(un[2 * kk + 1][2], un[2 * kk + 1][3]);
    }

    // O^T = S Qg^T + U_new^T P^T  [16 v x 64 t]
    float o[8][4];
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[a][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldb_nk_128(b, bufa + kStQg, 16 * np, 16 * kk, lane);
        mma_f16(o[2 * np], sa[kk], b[0], b[1]);
        mma_f16(o[2 * np + 1], sa[kk], b[2], b[3]);
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b[4];
        ldb_nk_64(b, bufa + kStP, 16 * np, 16 * kk, lane);
        mma_f16(o[2 * np], ua[kk], b[0], b[1]);
        mma_f16(o[2 * np + 1], ua[kk], b[2], b[3]);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t = 8 * j + 2 * q4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tt = t + (e & 1), vv = vl + 8 * (e >> 1);
        *reinterpret_cast<__nv_bfloat16*>(smem + kStO + swz64(tt, vv)) =
            __float2bfloat16_rn(o[j][e] * p.scale);
      }
    }

    // S = S Diag(gamma_C) + U_new^T K_hat
    const float* gc = reinterpret_cast<const float*>(buf + kStGc);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float g0 = gc[8 * j + 2 * q4], g1 = gc[8 * j + 2 * q4 + 1];
      s[j][0] *= g0; s[j][1] *= g1; s[j][2] *= g0; s[j][3] *= g1;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t b[4];
        ldb_kn_128(b, bufa + kStKh, 16 * np, 16 * kk, lane);
        mma_f16(s[2 * np], ua[kk], b[0], b[1]);
        mma_f16(s[2 * np + 1], ua[kk], b[2], b[3]);
      }
    }
    __syncthreads();

    // output rows t < L of this chunk (coalesced 16-byte stores)
    const int L = (int)min((int64_t)kChunk, len - ci * kChunk);
    const int64_t tok0 = bos + ci * kChunk;
    for (int idx = tid; idx < 64 * 8; idx += 128) {
      const int t = idx >> 3, ch = idx & 7;
      if (t < L) {
        const uint4 val = *reinterpret_cast<const uint4*>(smem + kStO + t * 128 + ((ch ^ (t & 7)) << 4));
        *reinterpret_cast<uint4*>(p.out + ((tok0 + t) * H + h) * kHeadDim + v0 + ch * 8) = val;
      }
    }
    if (ci + 2 < nch) load_chunk_operands(smem + cur * kStBuf, slot_ptr(ci + 2), v0, tid);
    cp_async_commit();
  }
  cp_async_wait<0>();

  // ---- final state ----
  if (p.final_state) {
    const int64_t sbase = (n * H + h) * (int64_t)(kHeadDim * kHeadDim);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int col = 8 * j + 2 * q4;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t off = sbase + (int64_t)(vr0 + 8 * hf) * kHeadDim + col;
        if (p.state_bf16)
          *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.final_state) + off) =
              pack_bf16(s[j][2 * hf], s[j][2 * hf + 1]);
        else
          *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.final_state) + off) =
              make_float2(s[j][2 * hf], s[j][2 * hf + 1]);
      }
    }
  }
}

void launch_state_kernel(const StateParams& p, cudaStream_t stream) {
  const int64_t blocks = p.N * p.H * 2;
  kda_state_kernel<<<(unsigned)blocks, 128, kStateSmem, stream>>>(p);
}

cudaError_t prepare_state_kernel() {
  return cudaFuncSetAttribute(kda_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kStateSmem);
}

}  // namespace kda
