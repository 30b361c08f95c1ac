// Token-by-token KDA forward: the fused_recurrent_kda entry point of the fla
// KDA code (fla-kda SKILL.md names chunk_kda and fused_recurrent_kda as the two
// public entry points).  Meant for decoding (one or a few tokens per sequence),
// where the chunked form has nothing to amortise: the cost is reading and
// writing the recurrent state, so the kernel is a streaming one.
//
// Per token, with S the state (row = value index, column = key index):
//   S' = S Diag(exp(a_t));  S = S' + beta (v - S' k) k^T;  o = scale S q
// (decay first, delta write with the decayed state, read-out after the write).
//
// One CTA per (sequence, head, 64-row value slab), 8 warps x 8 value rows;
// lane l holds key channels 4l .. 4l+3 of its warp's rows in fp32 registers for
// the whole sequence, so a row is one 512-byte access and the two dot products
// per row are warp shuffles.  Rows are independent, so the final state may be
// written over the initial one (each CTA reads its rows before writing them).
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

constexpr int kRecWarpRows = 8;                 // value rows per warp
constexpr int kRecRows = 8 * kRecWarpRows;       // value rows per CTA
constexpr int kRecThreads = 256;

__device__ __forceinline__ float rcp_fast(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(a) of one key channel: safe lb sigmoid(amul z), unsafe -amul softplus(z),
// or z itself already the log decay (same forms as the chunk kernel's gate).
template <int kGate>
__device__ __forceinline__ float rec_decay(float z, float amul, float lb) {
  if (kGate == kGateLogspace) return ex2(z * kLog2e);
  if (kGate == kGateUnsafe) return ex2(-amul * lg2(1.0f + ex2(z * kLog2e)));
  return ex2(lb * kLog2e * rcp_fast(1.0f + ex2(-amul * kLog2e * z)));
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ void load4_bf16(const uint16_t* p, float (&x)[4]) {
  const uint2 r = *reinterpret_cast<const uint2*>(p);
  const float2 a = unpack_bf16(r.x), b = unpack_bf16(r.y);
  x[0] = a.x;
  x[1] = a.y;
  x[2] = b.x;
  x[3] = b.y;
}

template <int kGate, bool kL2>
__global__ void __launch_bounds__(kRecThreads) kda_recurrent_kernel(RecurrentParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t H = p.H;
  const int slab = blockIdx.x % (kHeadDim / kRecRows);
  const int64_t unit = blockIdx.x / (kHeadDim / kRecRows);  // n * H + h
  const int64_t n = unit / H;
  const int h = (int)(unit - n * H);
  const int64_t bos = p.cu ? p.cu[n] : n * p.T;
  int64_t eos = p.cu ? p.cu[n + 1] : bos + p.T;
  if (p.cu) {  // bounds checked on the device: a sequence outside [0, T] is skipped
    const bool inside = bos >= 0 && eos >= bos && eos <= p.T;
    const bool bad = !inside || (n == 0 && bos != 0) || (n == p.N - 1 && eos != p.T);
    if (bad && threadIdx.x == 0 && p.status) atomicExch(p.status, 14);
    if (!inside) eos = bos;
  }
  const int c0 = 4 * lane;                        // key channels c0 .. c0 + 3
  const int r0 = slab * kRecRows + warp * kRecWarpRows;  // value rows r0 .. r0 + 7
  const int64_t sbase = unit * (int64_t)(kHeadDim * kHeadDim);

  float S[kRecWarpRows][4];
#pragma unroll
  for (int i = 0; i < kRecWarpRows; ++i) {
    const int64_t off = sbase + (int64_t)(r0 + i) * kHeadDim + c0;
    if (!p.init) {
      S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
    } else if (p.state_bf16) {
      load4_bf16(reinterpret_cast<const uint16_t*>(p.init) + off, S[i]);
    } else {
      const float4 x = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.init) + off);
      S[i][0] = x.x;
      S[i][1] = x.y;
      S[i][2] = x.z;
      S[i][3] = x.w;
    }
  }
  float dtb[4] = {0.f, 0.f, 0.f, 0.f};
  if (p.dt_bias && kGate != kGateLogspace) {
    const float4 x = *reinterpret_cast<const float4*>(p.dt_bias + h * kHeadDim + c0);
    dtb[0] = x.x;
    dtb[1] = x.y;
    dtb[2] = x.z;
    dtb[3] = x.w;
  }
  const float amul = (p.A_log && kGate != kGateLogspace) ? expf(p.A_log[h]) : 1.0f;

  for (int64_t t = bos; t < eos; ++t) {
    const int64_t row = t * H + h;
    float q[4], k[4], g[4], v[kRecWarpRows];
    load4_bf16(p.q + row * kHeadDim + c0, q);
    load4_bf16(p.k + row * kHeadDim + c0, k);
    if (p.g32) {
      const float4 x = *reinterpret_cast<const float4*>(p.g32 + row * kHeadDim + c0);
      g[0] = x.x;
      g[1] = x.y;
      g[2] = x.z;
      g[3] = x.w;
    } else {
      load4_bf16(p.g + row * kHeadDim + c0, g);
    }
    load4_bf16(p.v + row * kHeadDim + r0, *reinterpret_cast<float(*)[4]>(v));
    load4_bf16(p.v + row * kHeadDim + r0 + 4, *reinterpret_cast<float(*)[4]>(v + 4));
    const float braw = bf16_to_f(p.beta[row]);
    const float beta = p.beta_prob ? braw : rcp_fast(1.0f + ex2(-braw * kLog2e));
    if (kL2) {
      const float rq = rsqrtf(warp_sum(q[0] * q[0] + q[1] * q[1] + q[2] * q[2] + q[3] * q[3]) + 1e-6f);
      const float rk = rsqrtf(warp_sum(k[0] * k[0] + k[1] * k[1] + k[2] * k[2] + k[3] * k[3]) + 1e-6f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        q[c] *= rq;
        k[c] *= rk;
      }
    }
    float d[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) d[c] = rec_decay<kGate>(g[c] + dtb[c], amul, p.lower_bound);
    // decay, then the prediction S' k of each row
    float pr[kRecWarpRows];
#pragma unroll
    for (int i = 0; i < kRecWarpRows; ++i) {
      pr[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        S[i][c] *= d[c];
        pr[i] += S[i][c] * k[c];
      }
    }
#pragma unroll
    for (int i = 0; i < kRecWarpRows; ++i) pr[i] = warp_sum(pr[i]);
    // delta write, then the read-out S q
    float o[kRecWarpRows];
#pragma unroll
    for (int i = 0; i < kRecWarpRows; ++i) {
      const float w = beta * (v[i] - pr[i]);
      o[i] = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        S[i][c] += w * k[c];
        o[i] += S[i][c] * q[c];
      }
    }
#pragma unroll
    for (int i = 0; i < kRecWarpRows; ++i) o[i] = warp_sum(o[i]);
    if (lane == 0)
      *reinterpret_cast<uint4*>(p.out + row * kHeadDim + r0) =
          make_uint4(pack_bf16(o[0] * p.scale, o[1] * p.scale), pack_bf16(o[2] * p.scale, o[3] * p.scale),
                     pack_bf16(o[4] * p.scale, o[5] * p.scale), pack_bf16(o[6] * p.scale, o[7] * p.scale));
  }
  if (p.final_state) {
#pragma unroll
    for (int i = 0; i < kRecWarpRows; ++i) {
      const int64_t off = sbase + (int64_t)(r0 + i) * kHeadDim + c0;
      if (p.state_bf16)
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.final_state) + off) =
            make_uint2(pack_bf16(S[i][0], S[i][1]), pack_bf16(S[i][2], S[i][3]));
      else
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.final_state) + off) =
            make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
    }
  }
}

template <int kGate, bool kL2>
static void launch_rec(const RecurrentParams& p, cudaStream_t stream) {
  const int64_t blocks = p.N * p.H * (kHeadDim / kRecRows);
  kda_recurrent_kernel<kGate, kL2><<<(unsigned)blocks, kRecThreads, 0, stream>>>(p);
}

void launch_recurrent_kernel(const RecurrentParams& p, cudaStream_t stream) {
  if (p.N * p.H == 0) return;
  const bool l2 = p.l2norm != 0;
  switch (p.gate_mode) {
    case kGateUnsafe:
      if (l2) launch_rec<kGateUnsafe, true>(p, stream);
      else launch_rec<kGateUnsafe, false>(p, stream);
      break;
    case kGateLogspace:
      if (l2) launch_rec<kGateLogspace, true>(p, stream);
      else launch_rec<kGateLogspace, false>(p, stream);
      break;
    default:
      if (l2) launch_rec<kGateSafe, true>(p, stream);
      else launch_rec<kGateSafe, false>(p, stream);
  }
}

cudaError_t prepare_recurrent_kernel() { return cudaSuccess; }

}  // namespace kda
