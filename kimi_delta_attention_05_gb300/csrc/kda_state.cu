// Recurrent stage of the KDA forward pass: one CTA per (sequence, head,
// 32-wide value tile), walking the chunks of its sequence in order.
//
// Per chunk, with S the state (rows = value index, columns = key index) at
// the chunk start and the intra-chunk quantities of the workspace slot:
//   U_new = U - W S^T                     (delta-rule correction, WY form)
//   O     = scale (Q_gamma S^T + P U_new)  (inter + intra read-out, fused as in
//                                          the chunk_o stage of the fla code map)
//   S     = S Diag(gamma_C) + U_new^T K_hat   (chunk_delta_h state update)
//
// Work split: the CTA holds two "slabs" of 16 value rows; each slab is worked
// by four warps.  Warp q of a slab computes U_new and O for tokens
// 16q..16q+15 and owns key columns 32q..32q+31 of S (fp32, in mma
// accumulator registers).  Per chunk the slab's warps exchange S and U_new
// as fp16 operand tiles in shared memory (double-buffered by chunk parity),
// so the sequential chain per chunk is 2 x 16 mma.sync per warp plus one
// slab barrier and two CTA barriers.  Operands are fp16 (11-bit
// significand) with fp32 accumulation; the state itself stays fp32.
#include "kda_common.cuh"
#include "kda_kernels.cuh"

namespace kda {

// one chunk's operands (per buffer): the workspace slot image [0, kSlotUt)
// followed by this CTA's U^T tile
constexpr int kStW = kSlotW;     // tile128 [64 t][128 k] fp16
constexpr int kStQg = kSlotQg;   // tile128 [64 t][128 k] fp16
constexpr int kStKh = kSlotKh;   // tile128 [64 t][128 k] fp16
constexpr int kStP = kSlotP;     // tile64 [64 t][64 s] fp16
constexpr int kStGc = kSlotGc;   // fp32 [128]
constexpr int kStUt = kSlotUt;   // tile64 [32 v][64 t] fp16
constexpr int kStBuf = kSlotUt + 4096;
constexpr int kStages = 3;                     // operand pipeline depth
// exchange tiles, output staging, barriers
constexpr int kStS = kStages * kStBuf;         // [2 slab][2 parity] tile128 [16][128] fp16
constexpr int kStUn = kStS + 4 * 4096;         // [2 slab][2 parity] tile64 [16][64] fp16
constexpr int kStO = kStUn + 4 * 2048;         // [8 warps][16 t][16 v] bf16 output staging
constexpr int kStBar = kStO + 8 * 512;         // full, empty (CTA), empty (cluster) per stage
constexpr int kStAbort = kStBar + 24 * kStages;
constexpr int kStateSmem = kStAbort + 16;
constexpr int kVTile = 32;

// Sticky device status: set to KDA_ERR_DEVICE_TIMEOUT (13) by a CTA that gave
// up waiting for its operand copies; read and cleared by kda_get_status.
__device__ int g_kda_status = 0;

// The four CTAs of a cluster are the four value tiles of one (sequence,
// head); they need the same W / q gamma / k_hat / P / gamma_C block per chunk.
// Each CTA's elected thread fetches one quarter of that block and multicasts
// it to all four, plus its own U^T tile, all completing on the stage's full
// mbarrier of every destination CTA (same offsets everywhere).
constexpr int kClusterCtas = 4;
constexpr int kShareQuarter = kSlotUt / kClusterCtas;
static_assert(kShareQuarter % 16 == 0, "multicast pieces must be 16-byte multiples");

__device__ __forceinline__ void issue_chunk_copy(uint32_t dbase, uint32_t bar,
                                                 const unsigned char* slot, int vt) {
  fence_proxy_async_smem();
  mbar_expect_tx(bar, (uint32_t)kStBuf);
  const uint32_t off = (uint32_t)vt * kShareQuarter;  // vt == rank in the cluster
  bulk_g2s_multicast(dbase + off, slot + off, (uint32_t)kShareQuarter, bar, 0xF);
  bulk_g2s(dbase + kStUt, slot + kSlotUt + vt * 4096, 4096u, bar);
}

__device__ __forceinline__ void slab_barrier(int slab) {
  asm volatile("bar.sync %0, 128;\n" ::"r"(1 + slab));
}

// 8 consumer warps (two slabs x four) + 1 producer warp that only moves data.
constexpr int kStateThreads = 288;

__global__ void __launch_bounds__(kStateThreads, 1) kda_state_kernel(StateParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int slab = warp >> 2, qd = warp & 3;
  const int64_t H = p.H;
  const int64_t unit = blockIdx.x >> 2;
  const int vt = blockIdx.x & 3;
  const int v0 = vt * kVTile;
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
  const uint32_t sb = smem_u32(smem);
  const int vrow = v0 + 16 * slab + g;  // value rows vrow and vrow + 8
  const int kc0 = 32 * qd;              // this warp's key columns kc0 .. kc0 + 31
  const int64_t sbase = (n * H + h) * (int64_t)(kHeadDim * kHeadDim);

  auto slot_ptr = [&](int64_t ci) {
    return p.ws + ((slot0 + ci) * H + h) * (int64_t)kSlotBytes;
  };
  const uint32_t full0 = sb + kStBar, empty0 = sb + kStBar + 8 * kStages;
  const uint32_t cempty0 = sb + kStBar + 16 * kStages;
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kStAbort);
  if (tid == 0) {
    for (int st = 0; st < kStages; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, 8);               // one arrival per consumer warp
      mbar_init(cempty0 + 8 * st, kClusterCtas);   // one arrival per CTA of the cluster
    }
    *s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  cluster_sync();  // every CTA's barriers exist before any multicast lands
  // A timed-out wait sets the device status and switches the CTA to skip all
  // further waits: it finishes with garbage but never hangs.
  auto wait_or_abort = [&](uint32_t bar, uint32_t parity) {
    if (*s_abort) return;
    if (!mbar_wait_bounded(bar, parity)) {
      atomicExch(&g_kda_status, 13);
      *s_abort = 1;
    }
  };
  if (warp == 8) {
    // ---- producer warp: one elected lane streams chunk operands through the stages ----
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t ci = 0; ci < nch; ++ci) {
        const int st = (int)(ci % kStages);
        if (ci >= kStages) {
          const uint32_t ph = (uint32_t)(((ci - kStages) / kStages) & 1);
          wait_or_abort(empty0 + 8 * st, ph);  // this CTA's eight warps released it
#pragma unroll
          for (int rk = 0; rk < kClusterCtas; ++rk)
            asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];\n" ::"r"(
                             mapa_cluster(cempty0 + 8 * st, rk))
                         : "memory");
          if (!*s_abort && !mbar_wait_cluster_bounded(cempty0 + 8 * st, ph)) {
            atomicExch(&g_kda_status, 13);
            *s_abort = 1;
          }
        }
        if (*s_abort) break;
        issue_chunk_copy(sb + st * kStBuf, full0 + 8 * st, slot_ptr(ci), vt);
        issued = ci + 1;
      }
      // after a timeout, let this CTA's own issued copies land before leaving
      if (*s_abort)
        for (int64_t c = 0; c < issued; ++c)
          mbar_wait_bounded(full0 + 8 * (int)(c % kStages), (uint32_t)((c / kStages) & 1));
    }
    __syncwarp();
    cluster_sync();
    return;
  }
  // ---- initial state: s[nt] covers columns kc0 + 8 nt .. + 7 ----
  float s[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int col = kc0 + 8 * nt + 2 * q4;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      float x0 = 0.f, x1 = 0.f;
      if (p.init) {
        const int64_t off = sbase + (int64_t)(vrow + 8 * hf) * kHeadDim + col;
        float2 f;
        if (p.state_bf16)
          f = unpack_bf16(*reinterpret_cast<const uint32_t*>(
              reinterpret_cast<const uint16_t*>(p.init) + off));
        else
          f = *reinterpret_cast<const float2*>(reinterpret_cast<const float*>(p.init) + off);
        x0 = f.x;
        x1 = f.y;
      }
      s[nt][2 * hf] = x0;
      s[nt][2 * hf + 1] = x1;
    }
  }
  auto publish_state = [&](int par) {
    unsigned char* t = smem + kStS + (slab * 2 + par) * 4096;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        *reinterpret_cast<uint32_t*>(t + swz128(g + 8 * hf, kc0 + 8 * nt + 2 * q4)) =
            pack_f16(s[nt][2 * hf], s[nt][2 * hf + 1]);
  };
  publish_state(0);

  unsigned char* stage_o = smem + kStO + warp * 512;

  for (int64_t ci = 0; ci < nch; ++ci) {
    const int st = (int)(ci % kStages);
    const uint32_t ph = (uint32_t)((ci / kStages) & 1);
    const int par = (int)(ci & 1);
    const uint32_t bufa = sb + st * kStBuf;
    const unsigned char* buf = smem + st * kStBuf;
    const uint32_t Sa = sb + kStS + (slab * 2 + par) * 4096;
    const uint32_t Ua = sb + kStUn + (slab * 2 + par) * 2048;
    unsigned char* Un = smem + kStUn + (slab * 2 + par) * 2048;
    wait_or_abort(full0 + 8 * st, ph);
    slab_barrier(slab);  // S of this chunk (published by the slab's four warps) is visible

    // U_new^T [16 v x 16 t] = U^T - S W^T for tokens 16 qd .. 16 qd + 15
    uint32_t ut[4];  // U^T tile in accumulator layout (the A-fragment layout matches it)
    lda_64(ut, bufa + kStUt, 16 * slab, 16 * qd, lane);
    float x[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) x[a][b][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4], b[4];
      lda_128(a, Sa, 0, 16 * kk, lane);
      ldb_nk_128(b, bufa + kStW, 16 * qd, 16 * kk, lane);
      mma_f16(x[kk & 1][0], a, b[0], b[1]);
      mma_f16(x[kk & 1][1], a, b[2], b[3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int t = 16 * qd + 8 * nt + 2 * q4;
        const float2 u = unpack_f16(ut[2 * nt + hf]);
        const float n0 = u.x - (x[0][nt][2 * hf] + x[1][nt][2 * hf]);
        const float n1 = u.y - (x[0][nt][2 * hf + 1] + x[1][nt][2 * hf + 1]);
        *reinterpret_cast<uint32_t*>(Un + swz64(g + 8 * hf, t)) = pack_f16(n0, n1);
      }
    slab_barrier(slab);  // U_new of the slab is visible

    // S[:, kc0 ..] = S Diag(gamma_C) + U_new^T K_hat[:, kc0 ..]; publish for the next chunk
    const float* gc = reinterpret_cast<const float*>(buf + kStGc);
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float2 gg = *reinterpret_cast<const float2*>(gc + kc0 + 8 * nt + 2 * q4);
      s[nt][0] *= gg.x; s[nt][1] *= gg.y; s[nt][2] *= gg.x; s[nt][3] *= gg.y;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      lda_64(a, Ua, 0, 16 * kk, lane);
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b[4];
        ldb_kn_128(b, bufa + kStKh, kc0 + 16 * np, 16 * kk, lane);
        mma_f16(s[2 * np], a, b[0], b[1]);
        mma_f16(s[2 * np + 1], a, b[2], b[3]);
      }
    }
    publish_state(par ^ 1);

    // O^T [16 v x 16 t] = S Qg^T + U_new^T P^T for tokens 16 qd .. (S of the chunk start)
    float o[2][2][4];
#pragma unroll
    for (int a = 0; a < 2; ++a)
#pragma unroll
      for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[a][b][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4], b[4];
      lda_128(a, Sa, 0, 16 * kk, lane);
      ldb_nk_128(b, bufa + kStQg, 16 * qd, 16 * kk, lane);
      mma_f16(o[kk & 1][0], a, b[0], b[1]);
      mma_f16(o[kk & 1][1], a, b[2], b[3]);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4], b[4];
      lda_64(a, Ua, 0, 16 * kk, lane);
      ldb_nk_64(b, bufa + kStP, 16 * qd, 16 * kk, lane);
      mma_f16(o[kk & 1][0], a, b[0], b[1]);
      mma_f16(o[kk & 1][1], a, b[2], b[3]);
    }
    __syncwarp();
    if (lane == 0)  // release the stage (the producer forwards it to the cluster)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(empty0 + 8 * st) : "memory");
    // this warp's 16 x 16 output tile -> staging [16 t][16 v] -> 32-byte row segments
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tl = 8 * nt + 2 * q4 + (e & 1);
        const int vl = g + 8 * (e >> 1);
        *reinterpret_cast<__nv_bfloat16*>(stage_o + tl * 32 + vl * 2) =
            __float2bfloat16_rn((o[0][nt][e] + o[1][nt][e]) * p.scale);
      }
    __syncwarp();
    {
      const int L = (int)min((int64_t)kChunk, len - ci * kChunk);
      const int tl = lane >> 1, half = lane & 1;
      const int t = 16 * qd + tl;
      if (t < L) {
        const int64_t tok = bos + ci * kChunk + t;
        *reinterpret_cast<uint4*>(p.out + (tok * H + h) * kHeadDim + v0 + 16 * slab + 8 * half) =
            *reinterpret_cast<const uint4*>(stage_o + tl * 32 + half * 16);
      }
    }
    __syncwarp();
  }
  cluster_sync();  // no CTA leaves while others may still write into its shared memory

  // ---- final state ----
  if (p.final_state) {
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int col = kc0 + 8 * nt + 2 * q4;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int64_t off = sbase + (int64_t)(vrow + 8 * hf) * kHeadDim + col;
        if (p.state_bf16)
          *reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.final_state) + off) =
              pack_bf16(s[nt][2 * hf], s[nt][2 * hf + 1]);
        else
          *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.final_state) + off) =
              make_float2(s[nt][2 * hf], s[nt][2 * hf + 1]);
      }
    }
  }
}

extern "C" int kda_get_status(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_kda_status, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_kda_status, &z, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

void launch_state_kernel(const StateParams& p, cudaStream_t stream) {
  const int64_t blocks = p.N * p.H * (kHeadDim / kVTile);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kStateThreads);
  cfg.dynamicSmemBytes = kStateSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kda_state_kernel, p);
}

cudaError_t prepare_state_kernel() {
  return cudaFuncSetAttribute(kda_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kStateSmem);
}

}  // namespace kda
