// Recurrent stage of the KDA forward pass on the 5th-generation tensor cores
// (tcgen05, accumulators in tensor memory): one CTA per (sequence, head, value
// tile of 32 or 64 columns), walking the chunks of its sequence in order and
// bringing each chunk's operand block in with bulk copies, issued in parallel
// by nine lanes of a producer warp.  Four 32-column CTAs per head while they
// all fit on the GPU at once (shortest chunk period), else two 64-column ones
// (every CTA of a head receives the same 57 KB of chunk operands through its
// SM's L2 port, so fewer CTAs per head move fewer bytes).
//
// Per chunk, with S the state (rows = value index, columns = key index) at
// the chunk start and the intra-chunk quantities of the workspace slot:
//   U_new = U - W S^T                     (delta-rule correction, WY form)
//   O     = scale (Q_gamma S^T + P U_new)  (inter + intra read-out, fused as in
//                                          the chunk_o stage of the fla code map)
//   S     = S Diag(gamma_C) + U_new^T K_hat   (chunk_delta_h state update)
// as three tensor-core products, each issued by one elected lane of the
// tensor-core warp (widths for a tile of kVT value columns):
//   MMA1: D1 [128 x kVT] = [Q_gamma; W] (128 x 128) . S^T        (rows 64.. = W S^T)
//   MMA2: D3 [128 x kVT] = K_hat^T (128 x 64)       . U_new       (state delta, row = key)
//   MMA3: D1[0..63]     += [P; *]   (128 x 64)       . U_new       (output rows)
// The state master copy is fp32 in the registers of the epilogue warps
// (warp = tensor-memory lane quarter x 32-column group, thread = key index);
// each chunk it is published as an fp16 operand tile for the next MMA1.
// Roles: epilogue warps, then one bulk-copy warp, then the tensor-core warp.
// Waits on mbarriers (copies landed, products complete) are bounded: a CTA that
// gives up sets the device status word and stops waiting.  The two epilogue ->
// tensor-core hand-offs use named barriers, which every participating warp
// passes exactly once per chunk (plus once for the initial state) whatever
// happens, so they always complete.
#include "kda_common.cuh"
#include "kda_kernels.cuh"
#include "kda_tc.cuh"

namespace kda {

// ---- per-stage shared memory (one chunk's operands), 1024-aligned ----
constexpr int kSA1 = 0;          // kmaj R=128 K=128: [q gamma; W]
constexpr int kSKh = 32768;      // kmaj R=64 (t) K=128 (k): k_hat (MN-major A of MMA2)
constexpr int kSP = 49152;       // kmaj R=64 K=64: P  (rows 0..63 of the A operand of MMA3)
constexpr int kStages = 3;
// (U_new and S are published to the tensor-core warp through hardware named
// barriers, below: an mbarrier hand-off measured ~230-430 cycles, a named one
// ~120.)
constexpr int kBarFull = 0, kBarEmpty = 3, kBarMma1 = 6, kBarMma2 = 7, kBarMma3 = 8, kNumBars = 9;
constexpr int kPiece = kSP + 8192 - kSA1;    // 57344: the shared block minus gamma_C
constexpr int kPieces = 7;                   // copied as 7 pieces of 8 KB, one per lane
static_assert(kPiece == kPieces * 8192, "piece split");

// Layout and roles for a CTA of kVT value columns (32, 64 or 128; 128 / kVT
// CTAs per head).  Rows 64..127 of MMA3's A operand are the 8 KB after P:
// zeros with 32 columns; otherwise (where the zeros do not fit) whatever
// follows P, whose products land in rows of D1 that U_new has already consumed.
// (The layout also admits 128 columns, one head per SM: two stages of 73 KB
// and all 512 tensor-memory columns; its chunk period measured about twice
// the 32-column one, so no launch uses it.)
template <int kVT>
struct StateCfg {
  static constexpr int kVTile = kVT;
  static constexpr int kEpiWarps = 4 * (kVT / 32);  // (lane quarter, 32-column group) pairs
  static constexpr int kProducerWarp = kEpiWarps, kMmaWarp = kEpiWarps + 1;
  static constexpr int kThreads = 32 * (kEpiWarps + 2);
  static constexpr int kStg = kVT == 128 ? 2 : kStages;  // chunk stages in flight
  static constexpr bool kZeroPad = kVT == 32;
  static constexpr int kSZero = 57344;                   // 8 KB of zeros (kZeroPad only)
  static constexpr int kSGc = kZeroPad ? 65536 : 57344;  // fp32 [128] gamma_C
  static constexpr int kSU = kSGc + 512;                 // kVT / 32 U tiles [64 t][32 v] fp16
  static constexpr int kStageBytes = (kSU + kVT * 128 + 1023) / 1024 * 1024;
  static constexpr int kSS = kStg * kStageBytes;         // MN-major [128 k][kVT v] fp16: S
  static constexpr int kSUn = kSS + kVT * 256;           // MN-major [64 t][kVT v] fp16: U_new
  static constexpr int kSBar = kSUn + kVT * 128;         // mbarriers
  static constexpr int kSTmem = kSBar + 8 * kNumBars;    // tensor-memory base address
  static constexpr int kSAbort = kSTmem + 8;
  // 1 KB of slack after the last word: an operand read formed from any of the
  // descriptors above, under any swizzle mode, stays inside the allocation.
  static constexpr int kSmem = kSAbort + 8 + 1024;
  static constexpr uint32_t kStageTx = kPiece + 512 + kVT * 128;  // bytes landing per stage
  static constexpr uint32_t kTmemCols = kVT == 32 ? 128 : (kVT == 64 ? 256 : 512);  // D1 x 2, D3
  static constexpr int kNbSCount = 32 * (kEpiWarps + 1);       // S published: epilogue + MMA warp
  static constexpr int kNbUnCount = 32 * (kEpiWarps / 2 + 1);  // U_new published: lanes 64.. + MMA warp
  // The fp16 B operands S (N = v, K = k) and U_new (N = v, K = t) are stored
  // MN-major: one row of values per k (or t), so a thread that holds a row
  // writes it with 16-byte stores.  A row of a column block is one swizzle
  // atom wide: 64 columns (128-byte swizzle) or 32 (64-byte); 128 columns are
  // two 64-column blocks, the second `rows` rows after the first (the
  // descriptor's leading byte offset).
  static constexpr int kBlkCols = kVT < 64 ? kVT : 64;
  static constexpr int kRowB = 2 * kBlkCols;                 // bytes per row of a column block
  static constexpr uint32_t kBLayout = kVT == 32 ? 4u : 2u;  // descriptor: 64- / 128-byte swizzle
  static constexpr uint32_t kBSbo = 8 * kRowB;               // next group of 8 rows
  // byte offset of 16-byte chunk `chunk` (values 8 chunk .. 8 chunk + 7) of row `row` in a
  // tile of `rows` rows
  __device__ static uint32_t boff(int row, int chunk, int rows) {
    const int blk = chunk / (kBlkCols / 8), c = chunk % (kBlkCols / 8);
    return (uint32_t)(blk * rows * kRowB + row * kRowB +
                      ((c ^ (kVT == 32 ? ((row >> 1) & 3) : (row & 7))) << 4));
  }
  static_assert(kStageBytes % 1024 == 0 && kSS % 1024 == 0 && kSUn % 1024 == 0,
                "operand images need 1024-byte alignment");
  static_assert(kSU + kVT * 128 <= kStageBytes, "stage overflow");
  static_assert(kSmem <= 232448, "exceeds the opt-in shared memory of one CTA");
  static_assert(kStg <= kStages, "barrier slots");
};

// Hardware named barriers (ids 1, 2; 0 is __syncthreads): the publishing warps
// arrive, the tensor-core warp (all 32 lanes) waits.  Every participant passes
// each barrier the same number of times, whatever happens (no early exits).
constexpr int kNbS = 1, kNbUn = 2;
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

// kJobs: the CTA runs the job blockIdx.y of p.jobs (a chunk range with its own
// initial / final state, U possibly taken as zero, outputs possibly not
// written); without it, the ordinary run over every chunk.
template <int kVT, bool kJobs>
__global__ void __launch_bounds__(StateCfg<kVT>::kThreads, 1)
    kda_state_kernel(const __grid_constant__ StateParams p) {
  using C = StateCfg<kVT>;
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t H = p.H;
  constexpr int kTiles = kHeadDim / kVT;  // CTAs per head
  const int64_t unit = blockIdx.x / kTiles;
  const int vt = (int)(blockIdx.x % kTiles);
  const int v0 = vt * C::kVTile;
  const int64_t n = unit / H;
  const int h = (int)(unit - n * H);
  int64_t bos, len, slot0;
  int64_t nch;
  if (p.cu) {  // chunk count from the checked scan: 0 for a sequence with bad bounds
    bos = p.cu[n];
    len = p.cu[n + 1] - bos;
    slot0 = p.chunk_off[n];
    nch = p.chunk_off[n + 1] - slot0;
  } else {
    bos = n * p.ld;
    len = p.T;
    slot0 = n * p.NT;
    nch = (len + kChunk - 1) / kChunk;
  }
  // this CTA's run: a chunk range with its own initial and final state (job
  // fields other than the range and the two flags are read where they are used)
  const StateJob* job = kJobs ? &p.jobs[blockIdx.y] : nullptr;
  int64_t c_begin = 0, c_end = nch;
  bool u_zero = false, write_out = true;
  if (kJobs) {
    c_begin = min(job->c0, nch);
    c_end = min(job->c1, nch);
    u_zero = job->u_zero != 0;
    write_out = job->write_out != 0;
  }
  const int64_t ncj = c_end > c_begin ? c_end - c_begin : 0;  // chunks this CTA walks
  const uint32_t sb = smem_u32(smem);
  const uint32_t bar = sb + C::kSBar;
  auto B = [&](int i) { return bar + 8 * i; };
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + C::kSAbort);
  auto slot_ptr = [&](int64_t ci) {
    return p.ws + ((slot0 + ci) * H + h) * (int64_t)kSlotBytes;
  };

  // ---- set-up: barriers, zero tiles, tensor memory ----
  if (tid == 0) {
    for (int st = 0; st < C::kStg; ++st) {
      mbar_init(B(kBarFull + st), 1);
      mbar_init(B(kBarEmpty + st), 1 + C::kEpiWarps);  // MMA commit + the epilogue warps
    }
    mbar_init(B(kBarMma1), 1);
    mbar_init(B(kBarMma2), 1);
    mbar_init(B(kBarMma3), 1);
    *s_abort = (sb & 1023) ? 1 : 0;  // the swizzled operand images need 1024-byte alignment
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (C::kZeroPad)
    for (int i = tid; i < C::kStg * 512; i += C::kThreads)
      reinterpret_cast<uint4*>(smem + (i >> 9) * C::kStageBytes + C::kSZero)[i & 511] =
          make_uint4(0, 0, 0, 0);
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     sb + C::kSTmem),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kSTmem);
  if (*s_abort && tid == 0) atomicExch(p.status, 13);

  auto wait = [&](uint32_t b, uint32_t parity) {
    if (*s_abort) return;
    if (!mbar_wait_bounded(b, parity)) {
      atomicExch(p.status, 13);
      *s_abort = 1;
    }
  };

  if (warp == C::kProducerWarp) {
    // ---- bulk-copy producer: lane 0 keeps the barrier books, lanes 0..8 copy ----
    int64_t issued = 0;
    int st = 0;
    uint32_t ph_prev = 1;  // phase parity of the previous use of stage st
    for (int64_t it = 0; it < ncj; ++it) {
      const int64_t ci = c_begin + it;
      if (st == 0) ph_prev ^= 1u;
      if (it >= C::kStg) wait(B(kBarEmpty + st), ph_prev ^ 1u);  // the stage is free again
      __syncwarp();
      if (*s_abort) break;
      const uint32_t dst = sb + st * C::kStageBytes;
      const unsigned char* src = slot_ptr(ci);
      if (lane == 0) {
        fence_proxy_async_smem();
        mbar_expect_tx(B(kBarFull + st), C::kStageTx);
      }
      __syncwarp();
      if (lane < kPieces)
        bulk_g2s(dst + lane * 8192, src + lane * 8192, 8192u, B(kBarFull + st));
      else if (lane == kPieces)  // this CTA's two U tiles, adjacent in the slot
        bulk_g2s(dst + C::kSU, src + kSlotU + vt * (kVT * 128), kVT * 128u, B(kBarFull + st));
      else if (lane == kPieces + 1)
        bulk_g2s(dst + C::kSGc, src + kSlotGc, 512u, B(kBarFull + st));
      issued = it + 1;
      st = st + 1 == C::kStg ? 0 : st + 1;
    }
    // After a timeout: let the copies still in flight land before leaving.  Only
    // the last kStg can be: an earlier copy's stage was reused, so its own full
    // phase completed before the reuse was issued (and waiting on its parity
    // again could alias a later phase and spend the whole limit).
    if (*s_abort && lane == 0)
      for (int64_t c = issued > C::kStg ? issued - C::kStg : 0; c < issued; ++c)
        mbar_wait_bounded(B(kBarFull + (int)(c % C::kStg)), (uint32_t)((c / C::kStg) & 1));
  } else if (warp == C::kMmaWarp) {
    // ---- tensor-core issuer: the whole warp keeps step with the named barriers
    //      and runs the issue loops; one elected lane issues ----
    {
      const uint32_t id1 = idesc_f16(128, C::kVTile, false, true);
      const uint32_t id2 = idesc_f16(128, C::kVTile, true, true);
      const uint32_t d3 = tmem + 2 * C::kVTile;
      // descriptors of stage 0 / the fixed tiles; the 14-bit address field
      // (bytes >> 4) takes the stage and k-step offsets by plain addition
      const uint64_t dA1 = smem_desc(sb + kSA1, 16, 1024), dKh = smem_desc(sb + kSKh, 8192, 1024);
      const uint64_t dP = smem_desc(sb + kSP, 16, 1024);
      const uint64_t dS = smem_desc(sb + C::kSS, 128 * C::kRowB, C::kBSbo, C::kBLayout);
      const uint64_t dUn = smem_desc(sb + C::kSUn, 64 * C::kRowB, C::kBSbo, C::kBLayout);
      constexpr uint32_t kStepB = 16 * C::kRowB;  // one K step (16 rows) of an MN-major B
      int st = 0;
      uint32_t phf = 0;  // phase parity of the full barrier of stage st
      for (int64_t it = 0; it < ncj; ++it) {
        const uint32_t par = (uint32_t)(it & 1);
        const uint64_t so = (uint64_t)((st * C::kStageBytes) >> 4);
        const uint32_t d1 = tmem + C::kVTile * par;
        wait(B(kBarFull + st), phf);
        __syncwarp();  // bar.sync is warp-aligned: reconverge after the per-lane wait
        named_sync(kNbS, C::kNbSCount);  // S of this chunk published
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          tc_mma(d1, dA1 + so + (uint64_t)(((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                 dS + (uint64_t)((ks * kStepB) >> 4), id1, ks > 0);
        tc_commit(B(kBarMma1));
        named_sync(kNbUn, C::kNbUnCount);  // U_new of this chunk published
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(d3, dKh + so + (uint64_t)((ks * 2048) >> 4), dUn + (uint64_t)((ks * kStepB) >> 4),
                 id2, ks > 0);
        tc_commit(B(kBarMma2));  // the state update can start
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          tc_mma(d1, dP + so + (uint64_t)((ks * 32) >> 4), dUn + (uint64_t)((ks * kStepB) >> 4), id1, 1);
        tc_commit(B(kBarMma3));
        tc_commit(B(kBarEmpty + st));  // the stage's operands are no longer read by the tensor core
        if (++st == C::kStg) { st = 0; phf ^= 1u; }
      }
      named_sync(kNbS, C::kNbSCount);  // the state published after the last chunk (no product uses it)
      if (lane == 0 && ncj > 0)  // the last products must be complete before tensor memory is freed
        mbar_wait_bounded(B(kBarMma3), (uint32_t)((ncj - 1) & 1));
    }
  } else {
    // ---- epilogue warps 0-7: warp = (lane quarter q, column half hc); thread =
    //      tensor-memory lane (key index / token), 32 of the CTA's 64 value columns ----
    const int q = warp & 3, hc = warp >> 2;
    const int k = q * 32 + lane;  // 0..127
    const int vc = v0 + 32 * hc;  // first value column of this warp
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + 32 * hc;
    float s[32];  // S[vc + j][k], j = 0..31
    {
      const int64_t sbase = (n * H + h) * (int64_t)(kHeadDim * kHeadDim);
      const void* init = kJobs ? job->init : p.init;
      const int init_kind = kJobs ? job->init_kind : (p.init ? 1 : 0);
      const int init_bf16 = kJobs ? job->init_bf16 : p.init_bf16;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float x = 0.f;
        if (init_kind == 1) {
          const int64_t off = sbase + (int64_t)(vc + j) * kHeadDim + k;
          x = init_bf16 ? bf16_to_f(reinterpret_cast<const uint16_t*>(init)[off])
                        : reinterpret_cast<const float*>(init)[off];
        } else if (init_kind == 2) {
          x = (vc + j == k) ? 1.f : 0.f;
        }
        s[j] = x;
      }
    }
    auto publish_state = [&]() {  // row k of S^T: this warp's 32 values, four 16-byte chunks
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(smem + C::kSS + C::boff(k, 4 * hc + c, 128)) =
            make_uint4(pack_f16(s[8 * c], s[8 * c + 1]), pack_f16(s[8 * c + 2], s[8 * c + 3]),
                       pack_f16(s[8 * c + 4], s[8 * c + 5]), pack_f16(s[8 * c + 6], s[8 * c + 7]));
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      named_arrive(kNbS, C::kNbSCount);
    };
    publish_state();

    int st = 0;
    uint32_t phf = 0;
    for (int64_t it = 0; it < ncj; ++it) {
      const int64_t ci = c_begin + it;
      const uint32_t par = (uint32_t)(it & 1);
      const unsigned char* stg = smem + st * C::kStageBytes;
      wait(B(kBarFull + st), phf);
      const float gk = reinterpret_cast<const float*>(stg + C::kSGc)[k];
      if (q < 2) {  // gamma_C is all these warps read from the stage
        __syncwarp();
        if (lane == 0) mbar_arrive_local(B(kBarEmpty + st));
      }
      // U warps: this token's U row comes in before MMA1 completes (it landed with
      // the stage); the 128-column shape loads it after, within its register budget
      const int t = k - 64;  // token of this tensor-memory lane in rows 64.. of D1
      float uf[32];
      auto load_u = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(stg + C::kSU + hc * 4096 + utile_off(t, 8 * c));
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 uv = unpack_f16(uw[e]);
            uf[8 * c + 2 * e] = uv.x;
            uf[8 * c + 2 * e + 1] = uv.y;
          }
        }
      };
      if (kJobs && u_zero) {
#pragma unroll
        for (int j = 0; j < 32; ++j) uf[j] = 0.f;
      } else if (q >= 2 && kVT < 128) {
        load_u();
      }
      // only the U_new warps read MMA1's result now; the output rows wait for
      // MMA3 below (every suspending wait adds wake-up latency: 115 -> 110 us
      // on T=8192 H=32 without this one in the output warps)
      if (q >= 2) wait(B(kBarMma1), par);
      tc_fence_after();
      if (q >= 2) {
        if (kVT == 128 && !(kJobs && u_zero)) load_u();
        // U_new for token t: U - (W S^T)[t, :] (rows 64.. of D1)
        float x[32];
        tc_ld32(lane_addr + C::kVTile * par, x);
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // row t of U_new: this warp's 32 values
          uint32_t un[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * c + 2 * e;
            un[e] = pack_f16(uf[j] - x[j], uf[j + 1] - x[j + 1]);
          }
          *reinterpret_cast<uint4*>(smem + C::kSUn + C::boff(t, 4 * hc + c, 64)) =
              make_uint4(un[0], un[1], un[2], un[3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        named_arrive(kNbUn, C::kNbUnCount);
        if (lane == 0) mbar_arrive_local(B(kBarEmpty + st));  // U tile read
      }
      wait(B(kBarMma2), par);
      tc_fence_after();
      {
        // S[:, k] = gamma_C[k] S[:, k] + delta; publish for the next chunk
        float d[32];
        tc_ld32(lane_addr + 2 * C::kVTile, d);
#pragma unroll
        for (int j = 0; j < 32; ++j) s[j] = gk * s[j] + d[j];
        publish_state();
      }
      if (q < 2) {
        // output row t = k: D1 rows 0..63 = q gamma S^T + P U_new
        const int t = k;
        const int L = (int)min((int64_t)kChunk, len - ci * kChunk);
        float o[32];
        wait(B(kBarMma3), par);
        tc_fence_after();
        tc_ld32(lane_addr + C::kVTile * par, o);
        if ((!kJobs || write_out) && t < L) {
          const int64_t tok = bos + ci * kChunk + t;
          uint4* dst = reinterpret_cast<uint4*>(p.out + (tok * H + h) * kHeadDim + vc);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(pack_bf16(o[8 * c] * p.scale, o[8 * c + 1] * p.scale),
                                pack_bf16(o[8 * c + 2] * p.scale, o[8 * c + 3] * p.scale),
                                pack_bf16(o[8 * c + 4] * p.scale, o[8 * c + 5] * p.scale),
                                pack_bf16(o[8 * c + 6] * p.scale, o[8 * c + 7] * p.scale));
        }
        tc_fence_before();
      }
      if (++st == C::kStg) { st = 0; phf ^= 1u; }
    }
    // ---- final state ----
    void* fin = kJobs ? job->fin : p.final_state;
    const int fin_bf16 = kJobs ? job->fin_bf16 : p.final_bf16;
    if (fin) {
      const int64_t sbase = (n * H + h) * (int64_t)(kHeadDim * kHeadDim);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int64_t off = sbase + (int64_t)(vc + j) * kHeadDim + k;
        if (fin_bf16)
          reinterpret_cast<__nv_bfloat16*>(fin)[off] = __float2bfloat16_rn(s[j]);
        else
          reinterpret_cast<float*>(fin)[off] = s[j];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(C::kTmemCols));
}

template <int kVT>
static void launch_state_variant(const StateParams& p, cudaStream_t stream) {
  using C = StateCfg<kVT>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.N * p.H * (kHeadDim / kVT)), (unsigned)(p.njobs > 0 ? p.njobs : 1));
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  if (p.njobs > 0) cudaLaunchKernelEx(&cfg, kda_state_kernel<kVT, true>, p);
  else cudaLaunchKernelEx(&cfg, kda_state_kernel<kVT, false>, p);
}

// 32-column CTAs (four per head) give the shortest chunk period; 64-column
// CTAs (two per head) halve the bytes all CTAs of a head pull through their SM
// ports per chunk.  So: four per head while they fit on the GPU at once (one
// CTA per SM), two per head once they would run in more than one wave.
void launch_state_kernel(const StateParams& p, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t runs = p.N * p.H * (p.njobs > 0 ? p.njobs : 1);
  if (runs * 4 <= sms) launch_state_variant<32>(p, stream);
  else launch_state_variant<64>(p, stream);
}

// S_{g+1} = S_g M_g + R_g, fp32.  CTA (unit, row block) owns rows 16 rb .. 16 rb + 15
// of every S_g: a row of S_{g+1} needs only the same row of S_g, so the CTAs
// of a unit never wait for one another.  Thread = column c, rows 8 hr .. 8 hr + 7
// of the block; M is read column by column from global memory (L2), the rows
// of S_g from shared memory.
__global__ void __launch_bounds__(256) kda_split_combine_kernel(const float* X, const float* R,
                                                                const float* M, float* S,
                                                                int64_t units, int G) {
  __shared__ float rows[16][kHeadDim];
  const int64_t u = blockIdx.x;
  const int rb = blockIdx.y, c = threadIdx.x & 127, hr = threadIdx.x >> 7;
  constexpr int64_t kMat = (int64_t)kHeadDim * kHeadDim;
  for (int i = threadIdx.x; i < 16 * kHeadDim; i += 256)
    rows[i / kHeadDim][i % kHeadDim] = X[u * kMat + (16 * rb + i / kHeadDim) * kHeadDim + i % kHeadDim];
  __syncthreads();
  for (int g = 1; g + 1 < G; ++g) {
    const float* Mg = M + ((int64_t)(g - 1) * units + u) * kMat;
    const float* Rg = R + ((int64_t)(g - 1) * units + u) * kMat;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = Rg[(16 * rb + 8 * hr + i) * kHeadDim + c];
    for (int kk = 0; kk < kHeadDim; ++kk) {
      const float m = Mg[kk * kHeadDim + c];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(rows[8 * hr + i][kk], m, acc[i]);
    }
    __syncthreads();  // every thread has read rows of S_g
    float* Sg = S + ((int64_t)(g - 1) * units + u) * kMat;  // S_{g+1}
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      rows[8 * hr + i][c] = acc[i];
      Sg[(16 * rb + 8 * hr + i) * kHeadDim + c] = acc[i];
    }
    __syncthreads();
  }
}

void launch_split_combine(const float* X, const float* R, const float* M, float* S, int64_t units,
                          int G, cudaStream_t s) {
  if (G < 3 || units == 0) return;
  kda_split_combine_kernel<<<dim3((unsigned)units, 8), 256, 0, s>>>(X, R, M, S, units, G);
}

cudaError_t prepare_state_kernel() {
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(kda_state_kernel<32, false>, attr, StateCfg<32>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kda_state_kernel<64, false>, attr, StateCfg<64>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kda_state_kernel<32, true>, attr, StateCfg<32>::kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kda_state_kernel<64, true>, attr, StateCfg<64>::kSmem);
  return e;
}

}  // namespace kda
