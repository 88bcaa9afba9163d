// Launch arguments and launchers of the verification kernels (internal).
#pragma once

#include "common.cuh"

namespace sv {

struct ChainArgs {
  const char* target;
  const char* draft;
  const int32_t* tokens;
  const float* uniforms;                      // [B, k+1], or null: Philox per request
  const unsigned long long* seeds;            // [B] Philox keys (when uniforms is null)
  const unsigned long long* offsets;          // [B] Philox counters (when uniforms is null)
  const int32_t* draft_lens;                  // [B] real draft lengths (ragged), or null: k
  float c_hi, c_lo;  // log2(e)/T split as hi + lo
  float c_rn;        // log2(e)/T rounded to nearest (the bf16 one-fma exponents)
  int B, k, V;
  int rows;                    // logit rows per request in pass 1 (chain: 2k + 1; tree: N)
  int nvec, nsplit, vps;       // vectors per row, units per row, vectors per unit
  int nchunks, cpc, nsplit2;   // draw: chunks per row, per item, items per request
  int top_k;                   // filtered verify: tokens kept per row (0: no top-k)
  float top_p;                 // filtered verify: nucleus mass, in (0, 1]
  float min_p;                 // filtered verify: kept iff p >= min_p * max p (0: off)
  int wide;                    // filtered verify through per-row cuts (wide.cu): no top-k
                               // with top-p or min_p, or top_k > SPEC_MAX_TOPK
  int32_t* out_tokens;
  int32_t* out_n;
  float* out_probs;
  int32_t* seq_lens;
  long long wait_cycles;       // bound of every wait of the second phase (kWaitCycles)
  // stochastic tree verify: rows = N target rows per request (k = N - 1),
  // uniforms [B, N]
  const int32_t* tree_tokens;  // [B, N]
  const int32_t* paths;        // [B, P, L]
  int P, L;
  int32_t* out_best;           // [B] or null
  int32_t* out_nodes;          // [B, L] or null
  Ws ws;
};

struct ArgmaxArgs {
  const char* target;
  int B, R, V;                 // R rows per request (k+1 or N)
  int nvec, nsplit, vps;
  int tree;                    // 0: greedy chain, 1: tree
  const int32_t* draft_tokens; // greedy: [B, k]
  const int32_t* draft_lens;   // greedy: [B] real draft lengths (ragged), or null: k
  int k;
  const int32_t* tree_tokens;  // tree: [B, N]
  const int32_t* paths;        // tree: [B, P, L]
  int P, L;
  int32_t* out_tokens;
  int32_t* out_n;
  int32_t* out_best;
  int32_t* out_nodes;
  int32_t* seq_lens;
  long long wait_cycles;       // bound of every wait of the finish grid (kWaitCycles)
  Ws ws;
};

// Logit row r of request b in chain order: r <= k is target row r, r > k
// is draft row r-k-1.
__device__ __forceinline__ const char* row_ptr(const ChainArgs& a, int b, int r, size_t row_bytes) {
  return r <= a.k ? a.target + ((size_t)b * (a.k + 1) + r) * row_bytes
                  : a.draft + ((size_t)b * a.k + (r - a.k - 1)) * row_bytes;
}

// Whether row r of a request with the given draft length is verified: target
// rows 0..kb, draft rows 0..kb-1 (a length outside [0, k] verifies nothing).
__device__ __forceinline__ bool row_used(int k, int kb, int r) {
  if (kb < 0 || kb > k) return false;
  return r <= k ? r <= kb : r - k - 1 < kb;
}

// Enqueue the two chain passes (pass 2 as a programmatic dependent launch) /
// the argmax pass on `st`.  skip_pass1 (fault injection for tests only)
// launches the second grid alone, so that every word it waits for stays
// unwritten and each of its bounded waits runs out.
cudaError_t launch_chain(const ChainArgs& a, int dtype, bool vec, cudaStream_t st,
                         bool skip_pass1 = false);
cudaError_t launch_filtered(const ChainArgs& a, int dtype, bool vec, cudaStream_t st,
                            bool skip_pass1 = false);
cudaError_t launch_argmax(const ArgmaxArgs& a, int dtype, bool vec, cudaStream_t st,
                          bool skip_pass1 = false);
cudaError_t launch_tree_sampled(const ChainArgs& a, int dtype, bool vec, cudaStream_t st);
// Filtered chain verify with kept sets of any size (a.wide): six
// stream-ordered grids, nothing polls.
cudaError_t launch_wide(const ChainArgs& a, int dtype, bool vec, cudaStream_t st);

// Launch the first grid of a call as a programmatic dependent of whatever
// kernel precedes it on `st`: its CTAs may be scheduled while that grid's
// last CTAs finish, and it begins with griddepcontrol.wait, so it still runs
// after that grid has completed and sees all of its writes (stream order is
// kept; the next call's pass 1 no longer pays a full launch gap).
template <class Kern, class Arg>
cudaError_t launch_first(Kern kernel, long grid, int block, cudaStream_t st, const Arg& a) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Largest P * L of a stochastic tree verify (its paths and edge logits are
// staged in shared memory).
constexpr int kTreeStage = 4096;

// Host side of a chain verify (api.cu): argument checks that fill the
// launch arguments without writing anything, then the launch.
int chain_setup(ChainArgs& a, bool& vec, const void* target_logits, const void* draft_logits,
                int dtype, const int32_t* draft_tokens, const float* uniforms,
                const uint64_t* seeds, const uint64_t* offsets, const int32_t* draft_lens,
                float temperature, int B, int k, int V, int32_t* out_tokens,
                int32_t* out_num_accepted, float* out_probs, int32_t* seq_lens, void* workspace,
                size_t workspace_bytes, int top_k, float top_p, float min_p);
int chain_launch(const ChainArgs& a, int dtype, bool vec, cudaStream_t st, bool skip_pass1);

}  // namespace sv
