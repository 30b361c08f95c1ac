// Kernel parameter blocks and launch entry points shared by the host API.
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

struct kda_fwd_args;

namespace kda {

// Gate forms: lb sigmoid(exp(A_log) z), -exp(A_log) softplus(z), or g given as
// the log decay (no activation).
constexpr int kGateSafe = 0, kGateUnsafe = 1, kGateLogspace = 2;

// Intra-chunk stage (one CTA per (chunk slot, head)).
struct ChunkParams {
  const uint16_t *q, *k, *v, *g, *beta;  // bf16 [tokens, H, 128] / [tokens, H]
  const float* g32;                       // g as fp32 [tokens, H, 128], or nullptr (bf16 g)
  const float* A_log;                     // [H] or nullptr (safe gate only)
  const float* dt_bias;                   // [H, 128] or nullptr
  float lower_bound;
  int gate_mode;                          // kGateSafe / kGateUnsafe / kGateLogspace
  int beta_prob;                          // 1: beta holds beta itself, 0: logits
  int l2norm;
  const int64_t* cu;                      // [N+1] or nullptr (dense)
  const int64_t* chunk_off;               // [N+1] chunk prefix (varlen only)
  int64_t N, T, H;
  int64_t NT;                             // chunks per row (dense)
  int64_t ld;                             // dense: rows from one sequence's start to the next (>= T)
  unsigned char* ws;                      // first workspace slot
  int* status;                            // device status word (bounded waits that give up)
};

// One run of the recurrent stage over a chunk range of every sequence (dense
// calls only): initial state zero (kind 0), from a tensor (1) or the identity
// (2, which with U taken as zero makes the final state the range's transition
// matrix: S_end = S_start M + R is affine in S_start); final state written to
// `fin` if not null; outputs of the range written or not.
struct StateJob {
  int64_t c0, c1;       // chunk range [c0, c1) (clamped to each sequence's chunks)
  const void* init;     // [N, H, 128, 128] (kind 1)
  void* fin;            // [N, H, 128, 128] or nullptr
  int init_kind, init_bf16, fin_bf16;
  int u_zero;           // 1: U taken as zero
  int write_out;        // 1: write the range's outputs
};
constexpr int kMaxStateJobs = 16;

// Recurrent stage (one CTA per (sequence, head, value tile) and job).
struct StateParams {
  uint16_t* out;                          // bf16 [tokens, H, 128]
  const void* init;                       // [N, H, 128, 128] or nullptr
  void* final_state;                      // [N, H, 128, 128] or nullptr
  int init_bf16, final_bf16;              // state dtypes (1: bf16, 0: fp32)
  float scale;
  const int64_t* cu;
  const int64_t* chunk_off;
  int64_t N, T, H, NT;
  int64_t ld;                             // dense: rows from one sequence's start to the next (>= T)
  const unsigned char* ws;
  int* status;                            // status word of the caller's stream (waits that give up)
  int njobs;                              // 0: one run over every chunk with init / final_state
  StateJob jobs[kMaxStateJobs];           // else blockIdx.y selects one of njobs runs
};

// Token-by-token path (one CTA per (sequence, head, 32-row value slab)).
struct RecurrentParams {
  const uint16_t *q, *k, *v, *g, *beta;  // bf16 [tokens, H, 128] / [tokens, H]
  const float* g32;                       // g as fp32 [tokens, H, 128], or nullptr (bf16 g)
  uint16_t* out;                          // bf16 [tokens, H, 128]
  const float* A_log;
  const float* dt_bias;
  float lower_bound;
  float scale;
  int gate_mode;
  int beta_prob;
  int l2norm;
  const void* init;                       // [N, H, 128, 128] or nullptr
  void* final_state;                      // [N, H, 128, 128] or nullptr (may equal init)
  int state_bf16;
  const int64_t* cu;                      // [N+1] or nullptr (dense)
  int64_t N, T, H;
  int* status;                            // device status word (bad cu_seqlens)
};

// Host-side argument checks of kda_fwd (KDA_OK or an error code); on success
// the workspace slot count and the varlen header bytes.
int validate(const kda_fwd_args* args, int64_t* num_slots, size_t* header_bytes);

// Validate and enqueue one chunked forward pass on device buffers (the body
// of kda_fwd).  init_bf16 / final_bf16 >= 0 override the state dtype of the
// initial / final state separately (the host-buffer entry point carries the
// state between pieces in fp32 whatever the caller's dtype); -1 keeps
// args->state_dtype.  allow_split: the recurrent stage may run as a split
// pass over sequence segments when the policy picks one (needs the larger
// workspace that kda_fwd_workspace_bytes reports for such calls).
int fwd_device(const kda_fwd_args* args, void* workspace, size_t workspace_bytes,
               cudaStream_t stream, void* const* events, int init_bf16, int final_bf16,
               bool allow_split);

void launch_recurrent_kernel(const RecurrentParams& p, cudaStream_t s);
cudaError_t prepare_recurrent_kernel();
// Chunk prefix of packed sequences, checking 0 = cu[0] <= cu[1] <= ... <= cu[N] = T:
// a sequence whose bounds leave [0, T] or decrease gets no chunks, and any
// violation sets *status to 14 (KDA_ERR_BAD_SEQLENS).
void launch_chunk_offsets(const int64_t* cu, int64_t N, int64_t T, int64_t* chunk_off, int* status,
                          cudaStream_t s);
// Device address of the status word of stream `s` on the current device (a
// slot of the library's table, assigned on the stream's first use), or nullptr.
int* status_slot(cudaStream_t s);
// Persistent grid of two CTAs per SM (or fewer items); false if the inputs'
// tensor maps cannot be made (nothing launched).
bool launch_chunk_kernel(const ChunkParams& p, int64_t num_slots, cudaStream_t s);
// The 32-column shape (four CTAs per head) if all CTAs fit on the GPU at once
// (one per SM), else the 64-column one.
void launch_state_kernel(const StateParams& p, cudaStream_t s);
// Chains the segment transitions of a split pass for `units` (sequence, head)
// pairs: S_1 = X, S_{g+1} = S_g M_g + R_g for g = 1 .. G - 2, into S (S_2 .. S_{G-1});
// all fp32 [units][128][128], R and M indexed g - 1.
void launch_split_combine(const float* X, const float* R, const float* M, float* S, int64_t units,
                          int G, cudaStream_t s);
cudaError_t prepare_chunk_kernel();
cudaError_t prepare_state_kernel();

}  // namespace kda
