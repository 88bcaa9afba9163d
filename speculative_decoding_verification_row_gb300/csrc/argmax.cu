// Greedy verify: chain (Kestrel article 32, section 3.3: accept while the
// target's argmax equals the draft, emit the target's own token) and EAGLE
// tree (TensorRT-LLM deployment page, "Eagle-2" section: paths
// [batch, max_decoding_tokens, max_path_len]).
//
// Pass 1, argmax_kernel: one CTA per (request, row, unit) streams its slice
// of a target row once and keeps the first position of its largest stored
// value (compared exactly as fp32, lowest index on ties); it publishes the
// pair as one 64-bit word, never 0 (no fence, no counter).  Pass 2,
// argmax_finish_kernel, a programmatic dependent: one CTA per request waits
// for its words, merges the units of all rows, then either scans the chain
// (greedy) or walks every path of the tree, one path per thread, and keeps
// the longest accepted path.
#include "kernels.cuh"

namespace sv {

// A unit's (value, index) as one word: value bits low, index + 1 high, so a
// written word is never 0 and 0 means "not yet written".
__device__ __forceinline__ unsigned long long arg_pack(float v, int i) {
  return ((unsigned long long)(unsigned)(i + 1) << 32) | __float_as_uint(v);
}
__device__ __forceinline__ void arg_unpack(unsigned long long w, float& v, int& i) {
  v = __uint_as_float((uint32_t)w);
  i = (int)(uint32_t)(w >> 32) - 1;
}

// (value, index) order: larger value first, then lower index.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, off);
    const int oi = __shfl_xor_sync(0xffffffffu, i, off);
    if (better(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Fail-closed outputs of one request.
__device__ void argmax_fail(const ArgmaxArgs& a, int b) {
  const int W = a.tree ? a.L : a.k + 1;
  for (int i = threadIdx.x; i < W; i += kThreads) {
    a.out_tokens[(size_t)b * W + i] = -1;
    if (a.tree && a.out_nodes) a.out_nodes[(size_t)b * a.L + i] = -1;
  }
  if (threadIdx.x == 0) {
    a.out_n[b] = -1;
    if (a.tree && a.out_best) a.out_best[b] = -1;
    set_status(a.ws.status, SPEC_EBADINDEX);
  }
}

// Order-preserving key of a (value, index) pair: larger value, then lower
// index, compares larger as an unsigned integer.  -0 is taken as +0, as the
// float comparison does.
__device__ __forceinline__ unsigned long long arg_key(float v, int i) {
  uint32_t bits = v == 0.f ? 0u : __float_as_uint(v);
  bits = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
  return ((unsigned long long)bits << 32) | (uint32_t)~(uint32_t)i;
}
__device__ __forceinline__ int key_index(unsigned long long key) { return (int)~(uint32_t)key; }

// Largest tree a finish CTA stages in shared memory (paths of larger trees
// are read from global memory).
constexpr int kPathStage = 4096;

__device__ void argmax_epilogue(const ArgmaxArgs& a, int b) {
  __shared__ unsigned long long sKey[SPEC_MAX_TREE_NODES];  // per row: best (value, index)
  __shared__ int sTok[SPEC_MAX_TREE_NODES];                 // tree tokens / draft tokens
  __shared__ int sPaths[kPathStage];
  __shared__ int sBad;
  __shared__ int sAcc[kWarps], sPath[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int R = a.R, ns = a.nsplit;
  // Ragged greedy: kb <= k real drafts, rows 0..kb; a length outside [0, k]
  // fails closed.
  const int kraw = !a.tree && a.draft_lens ? a.draft_lens[b] : a.k;
  const bool bad_len = !a.tree && (kraw < 0 || kraw > a.k);
  const int kb = bad_len ? 0 : kraw;
  const int rows = a.tree ? R : (bad_len ? 0 : kb + 1);
  // Inputs first (they do not depend on pass 1).
  const int nt = a.tree ? R : a.k;
  const int32_t* tsrc = a.tree ? a.tree_tokens + (size_t)b * R : a.draft_tokens + (size_t)b * a.k;
  const int32_t* pb = a.tree ? a.paths + (size_t)b * a.P * a.L : nullptr;
  const bool staged = a.tree && a.P * a.L <= kPathStage;
  for (int i = threadIdx.x; i < nt; i += kThreads) sTok[i] = tsrc[i];
  if (staged)
    for (int i = threadIdx.x; i < a.P * a.L; i += kThreads) sPaths[i] = pb[i];
  for (int i = threadIdx.x; i < R; i += kThreads) sKey[i] = 0;
  if (threadIdx.x == 0) sBad = 0;
  __syncthreads();
  // Every unit word of the request, four loads in flight per thread, folded
  // into its row's key.  Pass 1 was scheduled in full before this grid, so
  // each wait ends; the bound turns a broken invariant into an error instead
  // of a hang.
  unsigned long long* words = reinterpret_cast<unsigned long long*>(a.ws.part) +
                              (size_t)b * R * ns;
  bool to = false;  // a wait of this thread ran out
  for (int i0 = threadIdx.x; i0 < rows * ns; i0 += 4 * kThreads) {
    unsigned long long w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * kThreads;
      w[q] = i < rows * ns ? ld_relaxed_u64(words + i) : 0;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * kThreads;
      if (i >= rows * ns) continue;
      if (!w[q]) {
        const long long t0 = clock64();
        while (!(w[q] = ld_relaxed_u64(words + i))) {
          if (clock64() - t0 > a.wait_cycles) {
            set_status(a.ws.status, SPEC_ETIMEOUT);
            w[q] = arg_pack(-INFINITY, 0);
            to = true;
            break;
          }
          __nanosleep(64);
        }
      }
      float v;
      int x;
      arg_unpack(w[q], v, x);
      atomicMax(&sKey[i / ns], arg_key(v, x));
    }
  }
  // A unit word that never arrived: the request fails closed.
  if (__syncthreads_or(to) && threadIdx.x == 0) sBad = 1;
  __syncthreads();
  // Every call leaves the workspace zero: clear this request's words.
  for (int i = threadIdx.x; i < R * ns; i += kThreads) words[i] = 0;

  if (!a.tree) {  // ---------------------------------------------- greedy chain
    const int k = a.k;
    if (threadIdx.x == 0 && bad_len) sBad = 1;
    for (int i = threadIdx.x; i < kb; i += kThreads)
      if (sTok[i] < 0 || sTok[i] >= a.V) sBad = 1;
    __syncthreads();
    if (sBad) {
      argmax_fail(a, b);
      return;
    }
    if (threadIdx.x == 0) {
      int j = 0;
      while (j < kb && key_index(sKey[j]) == sTok[j]) ++j;
      int32_t* out = a.out_tokens + (size_t)b * (k + 1);
      for (int i = 0; i <= k; ++i) out[i] = i < j ? sTok[i] : (i == j ? key_index(sKey[j]) : -1);
      a.out_n[b] = j;
      if (a.seq_lens) a.seq_lens[b] += j + 1;
    }
    return;
  }

  // --------------------------------------------------------------- tree
  const int N = R, P = a.P, L = a.L;
  const int32_t* paths = staged ? sPaths : pb;
  for (int n = threadIdx.x; n < N; n += kThreads)
    if (sTok[n] < 0 || sTok[n] >= a.V) sBad = 1;
  for (int e = threadIdx.x; e < P * L; e += kThreads) {
    const int32_t nd = paths[e];
    if (nd < -1 || nd >= N || (e % L == 0 && nd > 0)) sBad = 1;
  }
  __syncthreads();
  if (sBad) {
    argmax_fail(a, b);
    return;
  }
  // One path per thread; paths in increasing order so a strict '>' keeps the
  // lowest index among equally long paths.
  int best_acc = -1, best_p = INT_MAX;
  for (int p = threadIdx.x; p < P; p += kThreads) {
    const int32_t* path = paths + (size_t)p * L;
    if (path[0] < 0) continue;
    int acc = 0;
    for (int j = 1; j < L; ++j) {
      const int32_t node = path[j];
      if (node < 0 || sTok[node] != key_index(sKey[path[j - 1]])) break;
      ++acc;
    }
    if (acc > best_acc) {
      best_acc = acc;
      best_p = p;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const int oa = __shfl_xor_sync(0xffffffffu, best_acc, off);
    const int op = __shfl_xor_sync(0xffffffffu, best_p, off);
    if (oa > best_acc || (oa == best_acc && op < best_p)) {
      best_acc = oa;
      best_p = op;
    }
  }
  if (lane == 0) {
    sAcc[warp] = best_acc;
    sPath[warp] = best_p;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w)
      if (sAcc[w] > best_acc || (sAcc[w] == best_acc && sPath[w] < best_p)) {
        best_acc = sAcc[w];
        best_p = sPath[w];
      }
    const bool none = best_acc < 0;
    const int n = none ? 0 : best_acc;
    const int32_t* path = none ? nullptr : paths + (size_t)best_p * L;
    const int last = none ? 0 : path[n];
    int32_t* out = a.out_tokens + (size_t)b * L;
    for (int j = 0; j < L; ++j)
      out[j] = j < n ? sTok[path[j + 1]] : (j == n ? key_index(sKey[last]) : -1);
    if (a.out_nodes)
      for (int j = 0; j < L; ++j)
        a.out_nodes[(size_t)b * L + j] = j <= n ? (none ? 0 : path[j]) : -1;
    if (a.out_best) a.out_best[b] = none ? -1 : best_p;
    a.out_n[b] = n;
    if (a.seq_lens) a.seq_lens[b] += n + 1;
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 5) argmax_kernel(const ArgmaxArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched by launch_first
  asm volatile("griddepcontrol.launch_dependents;");
  using IO = Io<DT, VEC>;
  const int per_req = a.R * a.nsplit;
  const int b = blockIdx.x / per_req;
  const int rem = blockIdx.x - b * per_req;
  const int r = rem / a.nsplit;
  const int s = rem - r * a.nsplit;
  if (!a.tree && a.draft_lens) {  // ragged greedy: rows past the draft length are not verified
    const int kb = a.draft_lens[b];
    if (kb < 0 || kb > a.k || r > kb) return;
  }
  const char* row = a.target + ((size_t)b * a.R + r) * (size_t)a.V * IO::ES;
  const int vbeg = s * a.vps;
  const int vend = min(a.nvec, vbeg + a.vps);

  uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + (int)threadIdx.x + u * kThreads;
    if (v < vend) IO::load(row, v, w[u]);
  }
  // Largest value per vector; the first vector that reaches the thread's
  // maximum holds its first occurrence (vectors are visited in order).
  float best = -INFINITY;
  int bu = -1;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + (int)threadIdx.x + u * kThreads;
    if (v < vend) {
      const float vm = IO::vmax(w[u]);
      if (bu < 0 || vm > best) {
        best = vm;
        bu = u;
      }
    }
  }
  int idx = INT_MAX;
  if (bu >= 0) {
    uint32_t sel[IO::NW];
#pragma unroll
    for (int i = 0; i < IO::NW; ++i) sel[i] = w[0][i];
#pragma unroll
    for (int u = 1; u < kVecPerThread; ++u)
      if (u == bu)
#pragma unroll
        for (int i = 0; i < IO::NW; ++i) sel[i] = w[u][i];
    float e[IO::EPV];
    IO::unpack(sel, e);
    int first = 0;
#pragma unroll
    for (int i = IO::EPV - 1; i >= 0; --i)
      if (e[i] == best) first = i;
    idx = (vbeg + (int)threadIdx.x + bu * kThreads) * IO::EPV + first;
  }
  // Block reduce (value, index).
  __shared__ float sv_[kWarps];
  __shared__ int si_[kWarps];
  warp_argmax(best, idx);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sv_[warp] = best;
    si_[warp] = idx;
  }
  __syncthreads();
  if (warp == 0) {
    best = lane < kWarps ? sv_[lane] : -INFINITY;
    idx = lane < kWarps ? si_[lane] : INT_MAX;
    warp_argmax(best, idx);
    if (lane == 0)
      st_relaxed_u64(reinterpret_cast<unsigned long long*>(a.ws.part) + blockIdx.x,
                     arg_pack(best, idx));
  }
}

// One CTA per request (grid-stride).
__global__ void __launch_bounds__(kThreads) argmax_finish_kernel(const ArgmaxArgs a) {
  for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
    argmax_epilogue(a, b);
    __syncthreads();  // shared state of this request is no longer read
  }
  // Completion of this grid then implies completion of pass 1, which stream
  // order relies on (nothing above waits for the whole of pass 1).
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int DT, bool VEC>
cudaError_t launch_argmax_t(const ArgmaxArgs& a, cudaStream_t st, bool skip_pass1) {
  const long g = (long)a.B * a.R * a.nsplit;
  if (!skip_pass1) {
    const cudaError_t e = launch_first(argmax_kernel<DT, VEC>, g, kThreads, st, a);
    if (e != cudaSuccess) return e;
  }
  // Pass 2 may be scheduled once every pass-1 CTA has started.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.B < 1024 ? a.B : 1024));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, argmax_finish_kernel, a);
}

cudaError_t launch_argmax(const ArgmaxArgs& a, int dtype, bool vec, cudaStream_t st,
                          bool skip_pass1) {
  if (dtype == SPEC_BF16)
    return vec ? launch_argmax_t<SPEC_BF16, true>(a, st, skip_pass1)
               : launch_argmax_t<SPEC_BF16, false>(a, st, skip_pass1);
  return vec ? launch_argmax_t<SPEC_F32, true>(a, st, skip_pass1)
             : launch_argmax_t<SPEC_F32, false>(a, st, skip_pass1);
}

}  // namespace sv
