// Stochastic tree verify (TensorRT-LLM deployment page, "目标模型验证：树注意力与
// 批量并行": the EAGLE tree's tokens are judged against the target logits by
// rejection sampling; each level's children are chosen by top-K, "Eagle-2
// 多层级树状草稿生成").  Chosen children are point-mass proposals: at each node
// the children are tried in increasing node id, child c is accepted iff
// u[c] < p'(tok c), the current residual of the node's target row (a rejected
// child's token leaves the residual, which is renormalised), and when no child
// is accepted the final token is drawn from the residual by inverse CDF at
// u[0].  The emitted tokens then follow the target rows exactly.
//
// Pass 1 is chain_rowstats_kernel over the N target rows of each request.  The
// draw grid, a programmatic dependent, takes draw items (chunk ranges) of the
// request's final row.  Every item CTA stages the request's tree, gathers the
// logit of every tree edge (the child's token in its parent's row) before
// waiting on pass 1, merges the N rows' statistics in a fixed order, and walks
// the tree with one warp (each lane holds a bit per path on the accepted
// prefix; the next candidate is a warp minimum over those paths' next
// entries), so every item reaches the same node and rejected set.  It then sums
// the masked draw weights of its chunks, and the request's last item (atomic
// ticket) finds the token and writes the outputs.
#include <mutex>

#include "draw.cuh"

namespace sv {

namespace {

template <int DT, bool VEC>
__device__ __forceinline__ void tree_item(const ChainArgs& a, int b, int part) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  __shared__ float sM[SPEC_MAX_TREE_NODES], sS[SPEC_MAX_TREE_NODES];
  __shared__ int sTok[SPEC_MAX_TREE_NODES];
  __shared__ float sU[SPEC_MAX_TREE_NODES];
  __shared__ int sMask[SPEC_MAX_TREE_NODES];  // tokens rejected at the final node
  __shared__ short sPath[kTreeStage];
  __shared__ float sEdge[kTreeStage];  // [p * L + d]: logit of paths[p][d+1]'s token in row paths[p][d]
  __shared__ int sPrefix[SPEC_MAX_PATH_LEN];
  __shared__ unsigned sBits[SPEC_MAX_TREE_NODES / 32];  // the walk's candidate set
  __shared__ short sCandE[SPEC_MAX_TREE_NODES];        // a candidate's edge (index into sEdge)
  __shared__ int sLast, sFailed, sNode, sDepth, sNMask, sBest;
  __shared__ unsigned long long sWT[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = a.rows, P = a.P, L = a.L;
  const size_t row_bytes = (size_t)a.V * ES;
  const char* tb = a.target + (size_t)b * N * row_bytes;

  // Stage the tree and check it (inputs only, before the wait on pass 1).
  bool bad = false;
  for (int n = tid; n < N; n += kThreads) {
    const int t = a.tree_tokens[(size_t)b * N + n];
    bad |= t < 0 || t >= a.V;
    sTok[n] = t;
    sU[n] = a.uniforms[(size_t)b * N + n];
  }
  for (int e = tid; e < P * L; e += kThreads) {
    const int v = a.paths[(size_t)b * P * L + e];
    bad |= v < -1 || v >= N || (e % L == 0 && v > 0);
    sPath[e] = (short)v;  // a value out of range fails the request, unread
  }
  const bool any_bad = __syncthreads_or(bad);
  for (int e = tid; e < P * L; e += kThreads) {
    float x = -INFINITY;
    if (!any_bad && e % L < L - 1) {
      const int par = sPath[e], ch = sPath[e + 1];
      if (par >= 0 && ch >= 0) x = load_logit<DT>(tb + (size_t)par * row_bytes, sTok[ch]);
    }
    sEdge[e] = x;
  }

  // Merge the slice statistics of every row (all of them, also for a bad
  // request, so that its words are written before they are cleared): thread
  // r takes row r, issues the loads of all its words before using any
  // (waiting only for words still 0), then merges them in slice order.
  const unsigned long long* sb = a.ws.stats + (size_t)b * N * a.nsplit;
  bool to = false;  // a wait of this thread ran out
  for (int r = tid; r < N; r += kThreads) {
    const unsigned long long* pr = sb + (size_t)r * a.nsplit;
    float m = -INFINITY;
    for (int u0 = 0; u0 < a.nsplit; u0 += 16) {
      unsigned long long v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = u0 + q < a.nsplit ? ld_relaxed_u64(pr + u0 + q) : kNoStats;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (!v[q]) v[q] = wait_stats(a, pr + u0 + q, &to);  // only a present slice reads 0
        m = fmaxf(m, stats_unpack(v[q]).x);
      }
    }
    float sum = 0.f;
    if (m != -INFINITY)
      for (int u = 0; u < a.nsplit; ++u) {
        const float2 e = stats_unpack(ld_relaxed_u64(pr + u));  // written: seen above
        if (e.y > 0.f) sum += e.y * ex2(scaled(e.x - m, a.c_hi, a.c_lo));
      }
    sM[r] = m;
    sS[r] = sum;
  }
  // A statistics word that never arrived fails the request closed (the flag
  // reaches the finishing item through the ticket).
  const bool timed_out = __syncthreads_or(to);
  if (timed_out && tid == 0) atomicExch(&a.ws.sync[b].failed, 1);
  const bool skip = any_bad || timed_out;

  // The walk, in warp 0 (uniform across its lanes).  Lane l holds bit j for
  // path l + 32 j: set while the path's first d + 1 entries are the accepted
  // prefix.  At depth d the candidates are those paths' entries d + 1 (a
  // bitmap over node ids gives them in increasing id), tried 32 at a time:
  // lane i takes the i-th, with weight w_i = 2^(c(x - M)) of its edge logit
  // (0 when an earlier candidate at this node carried the same token, which
  // already left the residual), and S_rest before it is the row's S less the
  // weights of the candidates before it (all rejected if it is reached); the
  // first lane with u[c] < w_i / S_rest_i is the accepted child.
  if (warp == 0 && !skip) {
    unsigned long long alive = 0;
    for (int j = 0; j < (P + 31) / 32; ++j) {
      const int p = lane + 32 * j;
      if (p < P && sPath[p * L] == 0) alive |= 1ull << j;
    }
    const int nwords = (N + 31) / 32;
    int node = 0, d = 0, nmask = 0;
    if (lane == 0) sPrefix[0] = 0;
    while (d + 1 < L) {
      if (lane < nwords) sBits[lane] = 0u;
      __syncwarp();
      for (unsigned long long bits = alive; bits; bits &= bits - 1) {
        const int p = lane + 32 * (__ffsll((long long)bits) - 1);
        const int nx = sPath[p * L + d + 1];
        if (nx >= 0) {
          atomicOr(&sBits[nx >> 5], 1u << (nx & 31));
          sCandE[nx] = (short)(p * L + d);  // any alive path: the same edge logit
        }
      }
      __syncwarp();
      const unsigned word = lane < nwords ? sBits[lane] : 0u;
      const int cnt = __popc(word);
      int excl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, excl, o);
        if (lane >= o) excl += t;
      }
      const int total = __shfl_sync(0xffffffffu, excl, 31);
      excl -= cnt;
      const float M = sM[node];
      float Srest = sS[node];
      nmask = 0;
      int next = -1;
      for (int base = 0; base < total; base += 32) {
        const int idx = base + lane;
        int wsel = 0;  // the word holding candidate idx: the last with excl <= idx
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
          const int e = __shfl_sync(0xffffffffu, excl, wsel + step);
          if (wsel + step < nwords && e <= idx) wsel += step;
        }
        const unsigned wv = __shfl_sync(0xffffffffu, word, wsel);
        const int rank = idx - __shfl_sync(0xffffffffu, excl, wsel);
        const bool valid = idx < total;
        const int c = valid ? 32 * wsel + (int)__fns(wv, 0, rank + 1) : -1;
        const int tc = valid ? sTok[c] : -1;
        const unsigned same = __match_any_sync(0xffffffffu, valid ? tc : -2 - lane);
        bool gone = (same & ((1u << lane) - 1u)) != 0u;
        for (int i = 0; i < nmask && valid && !gone; ++i) gone = sMask[i] == tc;
        const float w = (valid && !gone) ? ex2(scaled(sEdge[sCandE[c]] - M, a.c_hi, a.c_lo)) : 0.f;
        float before = w;  // exclusive prefix of the weights
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, before, o);
          if (lane >= o) before += t;
        }
        const float batch = __shfl_sync(0xffffffffu, before, 31);
        before -= w;
        const float sr = Srest - before;
        const bool acc = valid && !gone && sr > 0.f && sU[c] < w / sr;
        const unsigned accm = __ballot_sync(0xffffffffu, acc);
        const int first = accm ? __ffs(accm) - 1 : 32;
        // the rejected candidates' tokens (before the accepted one) leave the residual
        const bool rej = valid && !gone && lane < first;
        const unsigned rejm = __ballot_sync(0xffffffffu, rej);
        if (rej) sMask[nmask + __popc(rejm & ((1u << lane) - 1u))] = tc;
        nmask += __popc(rejm);
        __syncwarp();
        if (accm) {
          next = __shfl_sync(0xffffffffu, c, first);
          break;
        }
        Srest -= batch;
      }
      if (next < 0) break;  // final draw at this node
      unsigned long long keep = 0;
      for (unsigned long long bits = alive; bits; bits &= bits - 1) {
        const int j = __ffsll((long long)bits) - 1;
        if (sPath[(lane + 32 * j) * L + d + 1] == next) keep |= 1ull << j;
      }
      alive = keep;
      ++d;
      node = next;
      nmask = 0;
      if (lane == 0) sPrefix[d] = next;
    }
    int bp = alive ? lane + 32 * (__ffsll((long long)alive) - 1) : INT_MAX;
    bp = __reduce_min_sync(0xffffffffu, bp);
    if (lane == 0) {
      sNode = node;
      sDepth = d;
      sNMask = nmask;
      sBest = bp == INT_MAX ? -1 : bp;
    }
  }
  __syncthreads();

  // This item's chunk sums of the final node's masked weights p(t) [t not in R].
  const int node = skip ? 0 : sNode;
  const char* prow = tb + (size_t)node * row_bytes;
  const float mp = skip ? 0.f : sM[node];
  const TokenMask mask{sMask, skip ? 0 : sNMask};
  if (!skip) {
    const int c0 = part * a.cpc, c1 = min(a.nchunks, c0 + a.cpc);
    const unsigned long long wt = chunk_sums<DT, VEC, true>(
        a, prow, nullptr, c0, c1, mp, 0.f, 0.f, a.ws.chunks + (size_t)b * a.nchunks, mask);
    if (lane == 0) sWT[warp] = wt;
    __syncthreads();
    if (tid == 0) {
      unsigned long long t = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += sWT[w];
      a.ws.items[(size_t)b * a.nsplit2 + part] = t;
    }
  }
  // One device-scope fence by thread 0 after the barrier releases the whole
  // CTA's sums (the fence is cumulative over the writes the barrier made
  // visible to it) before the ticket.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int t = atomicAdd(&a.ws.sync[b].tick2, 1);
    sLast = t == a.nsplit2 - 1;
    if (sLast) {
      a.ws.sync[b].tick2 = 0;
      __threadfence();
      sFailed = atomicExch(&a.ws.sync[b].failed, 0);
    }
  }
  __syncthreads();
  if (!sLast) return;

  // ---------------------------------------------------------- outputs
  for (int i = tid; i < N * a.nsplit; i += kThreads) const_cast<unsigned long long*>(sb)[i] = 0;
  int32_t* out = a.out_tokens + (size_t)b * L;
  if (skip || sFailed) {  // a bad token or node id, or a wait ran out: fail closed
    for (int i = tid; i < a.nchunks; i += kThreads) a.ws.chunks[(size_t)b * a.nchunks + i] = 0;
    for (int i = tid; i < a.nsplit2; i += kThreads) a.ws.items[(size_t)b * a.nsplit2 + i] = 0;
    for (int i = tid; i < L; i += kThreads) {
      out[i] = -1;
      if (a.out_nodes) a.out_nodes[(size_t)b * L + i] = -1;
    }
    if (tid == 0) {
      a.out_n[b] = -1;
      if (a.out_best) a.out_best[b] = -1;
      set_status(a.ws.status, SPEC_EBADINDEX);
    }
    return;
  }
  const int d = sDepth;
  const int tok = draw_token<DT, VEC, true>(a, b, prow, nullptr, mp, 0.f, 0.f, (double)sU[0], mask);
  for (int i = tid; i < L; i += kThreads) {
    out[i] = i < d ? sTok[sPrefix[i + 1]] : (i == d ? tok : -1);
    if (a.out_nodes) a.out_nodes[(size_t)b * L + i] = i <= d ? sPrefix[i] : -1;
  }
  if (tid == 0) {
    a.out_n[b] = d;
    if (a.out_best) a.out_best[b] = sBest;
    if (a.seq_lens) a.seq_lens[b] += d + 1;
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) tree_draw_kernel(const ChainArgs a) {
  const int items = a.B * a.nsplit2;
  for (int h = blockIdx.x; h < items; h += gridDim.x) {
    const int b = h / a.nsplit2;
    tree_item<DT, VEC>(a, b, h - b * a.nsplit2);
    __syncthreads();  // shared state of this item is no longer read
  }
  // Completion of this grid then implies completion of pass 1, which stream
  // order relies on.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int DT, bool VEC>
cudaError_t tree_slots(int* grid) {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tree_draw_kernel<DT, VEC>, kThreads, 0);
    if (e != cudaSuccess) return e;
    cached[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  *grid = cached[dev];
  return cudaSuccess;
}

template <int DT, bool VEC>
cudaError_t launch_tree_sampled_t(const ChainArgs& args, cudaStream_t st) {
  int slots = 0;
  cudaError_t e = tree_slots<DT, VEC>(&slots);
  if (e != cudaSuccess) return e;
  // Draw items of 64 chunks, doubled until the items fit in one wave, or
  // halved (down to 32) while twice as many still do: each item's chunk
  // sums are then one round of loads per warp.
  ChainArgs a = args;
  while ((long)a.B * a.nsplit2 > slots && a.cpc < a.nchunks) {
    a.cpc *= 2;
    a.nsplit2 = ceil_div(a.nchunks, a.cpc);
  }
  while (a.cpc > 32 && (long)a.B * ceil_div(a.nchunks, a.cpc / 2) <= slots) {
    a.cpc /= 2;
    a.nsplit2 = ceil_div(a.nchunks, a.cpc);
  }
  const long g1 = (long)a.B * a.rows * a.nsplit;
  e = launch_first(chain_rowstats_kernel<DT, VEC>, g1, kThreads, st, a);
  if (e != cudaSuccess) return e;
  const long items = (long)a.B * a.nsplit2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(items < slots ? items : slots));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_draw_kernel<DT, VEC>, a);
}

}  // namespace

cudaError_t launch_tree_sampled(const ChainArgs& a, int dtype, bool vec, cudaStream_t st) {
  if (dtype == SPEC_BF16)
    return vec ? launch_tree_sampled_t<SPEC_BF16, true>(a, st)
               : launch_tree_sampled_t<SPEC_BF16, false>(a, st);
  return vec ? launch_tree_sampled_t<SPEC_F32, true>(a, st)
             : launch_tree_sampled_t<SPEC_F32, false>(a, st);
}

}  // namespace sv
