// Accepted-KV relocation after a tree verify (TensorRT-LLM walkthrough, the
// "moving to the right place" step, _update_kv_cache_draft_token_location:
// the accepted nodes' rows, written in tree order during the draft step, are
// gathered into consecutive logical positions right after the committed
// prefix; the cache is paged).
//
// Request b's logical position t lives in pool row
// block_tables[b][t / tokens_per_block] * tokens_per_block + t % tokens_per_block.
// Row base + accepted_nodes[b][j] moves to row base + j for j = 1..n (node 0,
// the root, stays).  Along a path node_j >= j and nodes strictly increase, so
// copying in increasing j never reads a row an earlier copy wrote, nor
// overwrites a row a later copy reads: each thread can move its 16-byte
// column of the rows in place, eight rows at a time, with no barrier.
#include "kernels.cuh"

namespace sv {

namespace {

constexpr int kTile = kThreads * 16;  // bytes of a row one CTA moves
constexpr int kBatch = 8;             // rows in flight per thread

struct RelocArgs {
  char* pool;
  size_t row_bytes;
  int tpb, num_blocks, max_blocks;
  const int32_t* block_tables;
  const int32_t* base;
  const int32_t* nodes;
  const int32_t* num_accepted;
  int B, L;
};

// Pool row of logical position t of request b, or -1 when it is unmapped.
__device__ __forceinline__ long pool_row(const RelocArgs& a, int b, long t) {
  if (t < 0 || t >= (long)a.max_blocks * a.tpb) return -1;
  const int blk = a.block_tables[(size_t)b * a.max_blocks + t / a.tpb];
  if (blk < 0 || blk >= a.num_blocks) return -1;
  return (long)blk * a.tpb + t % a.tpb;
}

__global__ void __launch_bounds__(kThreads) relocate_kernel(const RelocArgs a) {
  const int b = blockIdx.y;
  const int n = a.num_accepted[b];
  if (n <= 0 || n >= a.L) return;  // nothing moves (or the request failed closed)
  const int32_t* nodes = a.nodes + (size_t)b * a.L;
  const long base = a.base[b];
  // Every CTA of the request checks the whole path, so they all agree on
  // whether the request moves at all: root first, strictly increasing nodes,
  // every source and destination mapped.
  __shared__ int sOk;
  if (threadIdx.x == 0) {
    int ok = nodes[0] == 0;
    for (int j = 1; j <= n && ok; ++j) {
      const int nd = nodes[j];
      ok = nd > nodes[j - 1] && pool_row(a, b, base + nd) >= 0 && pool_row(a, b, base + j) >= 0;
    }
    sOk = ok;
  }
  __syncthreads();
  if (!sOk) return;
  const size_t col = (size_t)blockIdx.x * kTile + (size_t)threadIdx.x * 16;
  if (col >= a.row_bytes) return;
  for (int j0 = 1; j0 <= n; j0 += kBatch) {
    uint4 v[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int j = j0 + q;
      if (j <= n && nodes[j] != j)
        v[q] = *reinterpret_cast<const uint4*>(a.pool + pool_row(a, b, base + nodes[j]) * a.row_bytes + col);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int j = j0 + q;
      if (j <= n && nodes[j] != j)
        *reinterpret_cast<uint4*>(a.pool + pool_row(a, b, base + j) * a.row_bytes + col) = v[q];
    }
  }
}

}  // namespace

}  // namespace sv

using namespace sv;

extern "C" int spec_relocate_accepted_kv(void* kv_pool, size_t row_bytes, int tokens_per_block,
                                         int num_blocks, const int32_t* block_tables,
                                         int max_blocks, const int32_t* base_lens,
                                         const int32_t* accepted_nodes,
                                         const int32_t* num_accepted, int B, int L,
                                         spec_stream_t stream) {
  if (!kv_pool || !block_tables || !base_lens || !accepted_nodes || !num_accepted)
    return SPEC_EINVAL;
  if (B < 1 || B > SPEC_MAX_BATCH || L < 1 || L > SPEC_MAX_PATH_LEN || tokens_per_block < 1 ||
      num_blocks < 1 || max_blocks < 1 || row_bytes == 0 || row_bytes % 16 != 0 ||
      reinterpret_cast<uintptr_t>(kv_pool) % 16 != 0)
    return SPEC_EINVAL;
  const size_t tiles = (row_bytes + kTile - 1) / kTile;
  if (tiles > 65535u * 1024u) return SPEC_EINVAL;
  RelocArgs a{static_cast<char*>(kv_pool), row_bytes, tokens_per_block, num_blocks, max_blocks,
              block_tables, base_lens, accepted_nodes, num_accepted, B, L};
  relocate_kernel<<<dim3((unsigned)tiles, (unsigned)B), kThreads, 0, (cudaStream_t)stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
