// Chain rejection-sampling verify on top-k / top-p filtered distributions
// (TensorRT-LLM walkthrough, rejection-sampling section: the target side is
// filtered by the same backend and parameters as the draft side was, or the
// accept test is silently wrong).  Every target and draft row is reduced to
// its kept set: the top_k tokens by (logit descending, token ascending), then
// the shortest prefix of them whose softmax mass (softmax over those top_k,
// at temperature T) reaches top_p, then those with 2^(c(x - x_max)) >= min_p;
// p and q are the softmax over the kept set.  This file serves
// 1 <= top_k <= SPEC_MAX_TOPK with explicit kept lists; wide.cu serves
// kept sets of any size (no top-k, or a larger one) through per-row cuts.
// The verify itself is the plain chain rule (vLLM anatomy page, "Speculative
// Decoding"): accept x_i iff r_i < p_i(x_i) / q_i(x_i) (q = 0 accepts), stop
// at the first rejection j and draw from max(0, p_j - q_j) normalised, or
// from p_k when all k are accepted.
//
// Two passes; every logit is read once from HBM, plus about K 128-byte lines
// per row.  A logit's key is (order-preserving bits of the logit) << 32 |
// (2^32 - 1 - token): larger key = larger logit, then lower token, so the
// kept set's order is the key order.  Logits of -inf are never kept: their
// weight is exactly 0, so they change no probability, no top-p prefix and no
// draw.
//   filter_max_kernel streams the rows like the unfiltered pass 1 and keeps
//   only one 16-bit code per 128 contiguous bytes (the prefix of its largest
//   logit's key).
//   filter_pick_kernel, one CTA per row, takes a code threshold that at
//   least K codes reach, re-reads only the 128-byte groups at or above it,
//   ranks their candidates and publishes the row's kept list (token,
//   probability) and the probability of the draft token the row tests; the
//   request's last row CTA (acquire-release ticket) runs the accept scan and
//   draws the final token by inverse CDF over the kept tokens of target row
//   j in token order (p_j is zero elsewhere): exact 64-bit fixed-point
//   weights, summed per token bucket to find the one holding u Z.
//   filter_row_kernel (rows too wide for one CTA's codes) streams each row
//   through one CTA with a running candidate threshold instead.
#include "kernels.cuh"

namespace sv {

namespace {

// The logit and the token of a make_key key.
__device__ __forceinline__ float key_value(unsigned long long key) {
  return unord32((uint32_t)(key >> 32));
}
__device__ __forceinline__ int key_token(unsigned long long key) {
  return (int)(0xffffffffu - (uint32_t)key);
}

// ------------------------------------------------------------------ per-row CTAs
// filter_row_kernel: one CTA of kRowThreads per logit row (target or draft).
// The row streams through registers in chunks of kRowThreads * kRowVecs
// 16-byte vectors, the next chunk loading while one is filtered.  Candidates
// are the logits whose key is >= kappa, a running threshold: at least K keys
// >= kappa are always held (or every finite logit seen, when fewer), so the
// row's top K are all candidates.  kappa starts from the first chunk's
// vector maxima and rises only when the candidate buffer would overflow (its
// keys are then cut to their exact top K).  After the last chunk the held
// keys are ranked; the top K get the softmax and the top-p cut.
constexpr int kRowThreads = 128;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowVecs = 4;                              // vectors per thread per chunk
constexpr int kChunkVecs = kRowThreads * kRowVecs;
constexpr int kBufCap = 1536;                            // candidate keys a row CTA holds
constexpr int kRankMax = 512;                            // final ranking without a cut first
constexpr int kRowCtasPerSm = 7;                         // 1064 rows resident on 152 SMs

struct RowSmem {
  unsigned long long buf[kBufCap + 2];   // held candidate keys (and a zero pad)
  alignas(16) unsigned long long top[SPEC_MAX_TOPK];  // the top K, sorted (cut / final
                                                      // ranking); the pick's stage
  unsigned long long kappa;              // candidates: key >= kappa
  int n;                                 // keys held
  int wsum[kRowWarps];                   // per-warp counts (scans)
  int red;                               // the drawn token (finish)
  uint32_t tcode;                        // threshold codes (warp minimum)
  float warp_f[kRowWarps];
  int m;                                 // top-p: kept entries
  float sm;                              // top-p: mass of the kept entries
  int last;                              // this CTA finishes the request
  int failed;                            // finish: a wait of the request ran out
};

// Block-wide sum of one int per thread over a kRowThreads CTA.
__device__ __forceinline__ int row_block_sum(int v, RowSmem& S) {
  const int w = (int)__reduce_add_sync(0xffffffffu, (unsigned)v);
  __syncthreads();  // earlier readers of S.wsum are done
  if ((threadIdx.x & 31) == 0) S.wsum[threadIdx.x >> 5] = w;
  __syncthreads();
  int t = 0;
#pragma unroll
  for (int q = 0; q < kRowWarps; ++q) t += S.wsum[q];
  return t;
}

// Exclusive block scan of one int per thread; *total gets the sum.
__device__ __forceinline__ int row_block_scan(int v, RowSmem& S, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();  // earlier readers of S.wsum are done
  if (lane == 31) S.wsum[warp] = incl;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int q = 0; q < kRowWarps; ++q) {
    const int t = S.wsum[q];
    before += q < warp ? t : 0;
    all += t;
  }
  *total = all;
  return before + incl - v;
}

// Rank the n held keys (unique): each key's rank is the number of keys above
// it; the top min(n, K) land in S.top in descending order.
__device__ void rank_held(RowSmem& S, int n, int K) {
  const int T = n <= kRowThreads / 4 ? 4 : n <= kRowThreads / 2 ? 2 : 1;
  const ulonglong2* kp = reinterpret_cast<const ulonglong2*>(S.buf);
  if (threadIdx.x == 0) S.buf[n] = 0;  // pads the last pair (0 is below every key)
  __syncthreads();
  for (int c0 = 0; c0 < n; c0 += kRowThreads / T) {
    const int ci = c0 + (int)threadIdx.x / T, part = (int)threadIdx.x % T;
    const unsigned long long key = ci < n ? S.buf[ci] : ~0ull;
    const int chunk = (((n + T - 1) / T) + 1) & ~1;
    const int q0 = part * chunk, q1 = min(n, q0 + chunk);
    int rank = 0;
#pragma unroll 4
    for (int q = q0; q < q1; q += 2) {
      const ulonglong2 kv = kp[q >> 1];
      rank += (kv.x > key ? 1 : 0) + (kv.y > key ? 1 : 0);
    }
    for (int o = 1; o < T; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (ci < n && part == 0 && rank < K) S.top[rank] = key;
  }
  __syncthreads();
}

// Sort the n held keys (unique, n <= kRowThreads * E) in descending order by
// a bitonic network over P = kRowThreads * E slots (the slots past n hold 0,
// below every key), thread t holding slots E t .. E t + E - 1; the top
// min(n, K) land in S.top.  Element i of a compare-exchange at distance j in
// merge stage kk keeps the larger of itself and i ^ j when (i & j) == 0
// equals (i & kk) == 0.  Partners within a thread are registers, within a
// warp shuffles, otherwise a round through S.buf.
template <int E, int J>
__device__ __forceinline__ void sort_local(unsigned long long (&v)[E], int base, int kk) {
#pragma unroll
  for (int e = 0; e < E; ++e)
    if ((e & J) == 0) {  // slot base + e is the lower of the pair
      const unsigned long long x = v[e], y = v[e | J];
      const bool big_first = ((base + e) & kk) == 0;
      v[e] = (x > y) == big_first ? x : y;
      v[e | J] = (x > y) == big_first ? y : x;
    }
}

template <int E>
__device__ __noinline__ void sort_held(RowSmem& S, int n, int K) {
  constexpr int P = kRowThreads * E;
  const int tid = threadIdx.x;
  unsigned long long v[E];
#pragma unroll
  for (int e = 0; e < E; ++e) v[e] = tid * E + e < n ? S.buf[tid * E + e] : 0ull;
  for (int kk = 2; kk <= P; kk <<= 1) {
    for (int j = kk >> 1; j > 0; j >>= 1) {
      if (j < E) {
        if (j == 1) sort_local<E, 1>(v, tid * E, kk);
        if constexpr (E >= 4)
          if (j == 2) sort_local<E, 2>(v, tid * E, kk);
      } else {
        unsigned long long o[E];
        if (j / E < 32) {
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = __shfl_xor_sync(0xffffffffu, v[e], j / E);
        } else {
          __syncthreads();  // earlier readers of S.buf are done
#pragma unroll
          for (int e = 0; e < E; ++e) S.buf[tid * E + e] = v[e];
          __syncthreads();
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] = S.buf[(tid * E + e) ^ j];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = tid * E + e;
          const bool keep_big = ((i & j) == 0) == ((i & kk) == 0);
          v[e] = (v[e] > o[e]) == keep_big ? v[e] : o[e];
        }
      }
    }
  }
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (tid * E + e < K) S.top[tid * E + e] = v[e];
  __syncthreads();
}

// Cut the held keys to their exact top K and raise kappa to the K-th key
// (n > K): the K-th largest key by bisection on its 64 bits (block-wide
// counts), then the K keys >= it move to the front of the buffer.
__device__ __noinline__ void cut_held(RowSmem& S, int K) {
  const int n = S.n;
  unsigned long long kth = 0;
  for (int bit = 63; bit >= 0; --bit) {
    const unsigned long long c = kth | (1ull << bit);
    int cnt = 0;
    for (int i = threadIdx.x; i < n; i += kRowThreads) cnt += S.buf[i] >= c ? 1 : 0;
    if (row_block_sum(cnt, S) >= K) kth = c;
  }
  // exactly K keys are >= kth (keys are unique): gather them in S.top at
  // scanned offsets, then back to the front of the buffer
  int mine = 0;
  for (int i = threadIdx.x; i < n; i += kRowThreads) mine += S.buf[i] >= kth ? 1 : 0;
  int total;
  int off = row_block_scan(mine, S, &total);
  for (int i = threadIdx.x; i < n; i += kRowThreads)
    if (S.buf[i] >= kth) S.top[off++] = S.buf[i];
  __syncthreads();
  for (int i = threadIdx.x; i < total; i += kRowThreads) S.buf[i] = S.top[i];
  if (threadIdx.x == 0) {
    S.n = total;
    S.kappa = kth;
  }
  __syncthreads();
}

// Raise kappa cheaply (n held keys, n > 4K): warp w takes keys w, w + 4, ...
// and finds the cw-th largest 16-bit prefix of their order bits (cw =
// ceil(K / 4), bisection between its least and largest); the least of the
// four, as a key prefix, keeps at least K keys.  The keys below it go.
__device__ __noinline__ void raise_held(RowSmem& S, int K) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = S.n;
  const int cw = (K + kRowWarps - 1) / kRowWarps;
  uint32_t lo = ~0u, hi = 0;
  for (int i = warp + kRowWarps * lane; i < n; i += kRowThreads) {
    const uint32_t p = (uint32_t)(S.buf[i] >> 48);
    lo = min(lo, p);
    hi = max(hi, p);
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  while (lo < hi) {  // every key of the share is >= lo, and the share holds >= cw keys
    const uint32_t mid = (lo + hi + 1) >> 1;
    unsigned c = 0;
    for (int i = warp + kRowWarps * lane; i < n; i += kRowThreads)
      c += (uint32_t)(S.buf[i] >> 48) >= mid ? 1u : 0u;
    if ((int)__reduce_add_sync(0xffffffffu, c) >= cw) lo = mid;
    else hi = mid - 1;
  }
  if (lane == 0) atomicMin(&S.tcode, lo);
  __syncthreads();
  const unsigned long long kap = (unsigned long long)S.tcode << 48;
  int mine = 0;
  for (int i = tid; i < n; i += kRowThreads) mine += S.buf[i] >= kap ? 1 : 0;
  int total;
  int off = row_block_scan(mine, S, &total);
  // Gather the survivors in order into S.top-sized pieces is not possible
  // (they may be more than SPEC_MAX_TOPK), so move them within the buffer:
  // every key is read before any is written.
  unsigned long long keep[kBufCap / kRowThreads];
#pragma unroll
  for (int q = 0; q < kBufCap / kRowThreads; ++q) {
    const int i = tid + q * kRowThreads;
    keep[q] = i < n ? S.buf[i] : 0ull;
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < kBufCap / kRowThreads; ++q)
    if (keep[q] >= kap && keep[q] != 0ull) S.buf[off++] = keep[q];
  if (tid == 0) {
    S.n = total;
    if (kap > S.kappa) S.kappa = kap;
    S.tcode = ~0u;
  }
  __syncthreads();
}

// Exclusive block scan of one float per thread (kRowThreads CTA).
__device__ __forceinline__ float row_block_scan_f(float v, RowSmem& S, float* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();
  if (lane == 31) S.warp_f[warp] = incl;
  __syncthreads();
  float before = 0.f, all = 0.f;
#pragma unroll
  for (int q = 0; q < kRowWarps; ++q) {
    const float t = S.warp_f[q];
    before += q < warp ? t : 0.f;
    all += t;
  }
  *total = all;
  return before + incl - v;
}

__device__ __forceinline__ unsigned long long* row_words_of(const ChainArgs& a, int b, int r) {
  return a.ws.cand + ((size_t)b * (2 * a.k + 1) + r) * (size_t)a.top_k;
}

__device__ void finish_request(RowSmem& S, const ChainArgs& a, int b);

// Chunk c of a row into registers (thread t: vectors c * kChunkVecs + t +
// u * kRowThreads).
template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(const char* row, int c, int nvec,
                                           uint32_t (&X)[kRowVecs][Io<DT, VEC>::NW]) {
#pragma unroll
  for (int u = 0; u < kRowVecs; ++u) {
    const int v = c * kChunkVecs + (int)threadIdx.x + u * kRowThreads;
    if (v < nvec) Io<DT, VEC>::load(row, v, X[u]);
  }
}

// The candidates among the logits of vector v (register form w): logits
// x > -inf with key >= kap; emit(key) for each, in order.
template <int DT, bool VEC, typename F>
__device__ __forceinline__ void vec_candidates(int v, const uint32_t (&w)[Io<DT, VEC>::NW],
                                               unsigned long long kap, F emit) {
  constexpr int EPV = Io<DT, VEC>::EPV;
  float e[EPV];
  Io<DT, VEC>::unpack(w, e);
#pragma unroll
  for (int q = 0; q < EPV; ++q)
    if (e[q] > -INFINITY) {
      const unsigned long long key = make_key(e[q], (long)v * EPV + q);
      if (key >= kap) emit(key);
    }
}

// Append the candidates of this thread's vectors vidx[u] (register form
// X[u], maxima vm[u]; cnt candidates in all) to the held keys.
template <int DT, bool VEC, int NV>
__device__ __forceinline__ void append_chunk(RowSmem& S, int K, const int (&vidx)[NV],
                                             const uint32_t (&X)[NV][Io<DT, VEC>::NW],
                                             const float (&vm)[NV], int cnt) {
  const int tid = threadIdx.x;
  unsigned long long kap = S.kappa;
  float kv = kap ? key_value(kap) : -INFINITY;
  int total;
  int off = row_block_scan(cnt, S, &total);
  if (S.n + total <= kBufCap) {  // all of the chunk's candidates fit
    unsigned long long* dst = S.buf + S.n + off;
#pragma unroll
    for (int u = 0; u < NV; ++u)
      if (vm[u] >= kv && vm[u] > -INFINITY)
        vec_candidates<DT, VEC>(vidx[u], X[u], kap, [&](unsigned long long key) { *dst++ = key; });
    __syncthreads();
    if (tid == 0) S.n += total;
    __syncthreads();
    if (S.n > max(4 * K, 256)) raise_held(S, K);
    return;
  }
  // Vector by vector, cutting the held keys to the top K first when the
  // vector's candidates (at most kRowThreads * EPV) would not fit.
#pragma unroll
  for (int u = 0; u < NV; ++u) {
    const int v = vidx[u];
    for (int attempt = 0; attempt < 2; ++attempt) {
      kap = S.kappa;
      kv = kap ? key_value(kap) : -INFINITY;
      int cu = 0;
      if (vm[u] >= kv && vm[u] > -INFINITY)
        vec_candidates<DT, VEC>(v, X[u], kap, [&](unsigned long long) { ++cu; });
      off = row_block_scan(cu, S, &total);
      if (S.n + total > kBufCap && attempt == 0) {  // then S.n > kBufCap - kRowThreads * 8 > K
        cut_held(S, K);
        continue;
      }
      unsigned long long* dst = S.buf + S.n + off;
      if (vm[u] >= kv && vm[u] > -INFINITY)
        vec_candidates<DT, VEC>(v, X[u], kap, [&](unsigned long long key) { *dst++ = key; });
      __syncthreads();
      if (tid == 0) S.n += total;
      __syncthreads();
      break;
    }
  }
}

// Filter chunk c (in registers): its candidates join the held keys.  The
// first chunk also sets kappa0: each warp's cw-th largest vector maximum
// (16-bit prefix of the order bits, bisection between the warp's least and
// largest), the least over the warps, so at least K logits are >= it.  0:
// some warp has fewer than cw finite vectors (every finite logit counts).
template <int DT, bool VEC>
__device__ __forceinline__ void filter_chunk(RowSmem& S, int K, int c, int nvec,
                                             const uint32_t (&X)[kRowVecs][Io<DT, VEC>::NW]) {
  const int tid = threadIdx.x, lane = tid & 31;
  float vm[kRowVecs];
  int vidx[kRowVecs];
#pragma unroll
  for (int u = 0; u < kRowVecs; ++u) {
    vidx[u] = c * kChunkVecs + tid + u * kRowThreads;
    vm[u] = vidx[u] < nvec ? Io<DT, VEC>::vmax(X[u]) : -INFINITY;
  }
  if (c == 0) {
    const int cw = (K + kRowWarps - 1) / kRowWarps;
    uint32_t mo[kRowVecs], lo = ~0u, hi = 0;
#pragma unroll
    for (int u = 0; u < kRowVecs; ++u) {
      mo[u] = vm[u] > -INFINITY ? ord32(vm[u]) >> 16 : 0u;
      lo = min(lo, mo[u]);
      hi = max(hi, mo[u]);
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    while (lo < hi) {  // all 128 of the warp's maxima are >= lo, and cw <= 64
      const uint32_t mid = (lo + hi + 1) >> 1;
      unsigned n = 0;
#pragma unroll
      for (int u = 0; u < kRowVecs; ++u) n += mo[u] >= mid ? 1u : 0u;
      if ((int)__reduce_add_sync(0xffffffffu, n) >= cw) lo = mid;
      else hi = mid - 1;
    }
    if (lane == 0) atomicMin(&S.tcode, lo << 16);
    __syncthreads();
    if (tid == 0) {
      S.kappa = (unsigned long long)S.tcode << 32;
      S.tcode = ~0u;  // for raise_held
    }
    __syncthreads();
  }
  const unsigned long long kap = S.kappa;
  const float kv = kap ? key_value(kap) : -INFINITY;
  int cnt = 0;
#pragma unroll
  for (int u = 0; u < kRowVecs; ++u)
    if (vm[u] >= kv && vm[u] > -INFINITY)
      vec_candidates<DT, VEC>(vidx[u], X[u], kap, [&](unsigned long long) { ++cnt; });
  if (__syncthreads_or(cnt > 0)) append_chunk<DT, VEC, kRowVecs>(S, K, vidx, X, vm, cnt);
}

// The row's candidates are held: rank them, softmax and top-p cut over the
// top K, and publish the kept list (token, probability) and the probability
// of the draft token this row tests.
__device__ __forceinline__ void publish_row(RowSmem& S, const ChainArgs& a, int b, int r, int kb) {
  const int tid = threadIdx.x;
  const int K = a.top_k, k = a.k;
  int n = S.n;
  if (n > kRankMax) {
    cut_held(S, K);
    n = S.n;
  }
  if (n <= kRowThreads) rank_held(S, n, K);
  else if (n <= 2 * kRowThreads) sort_held<2>(S, n, K);
  else sort_held<4>(S, n, K);
  const int kk = min(n, K);  // real keys in S.top

  // Softmax over the top K at temperature T, then the top-p cut; thread t
  // holds entries 2t and 2t + 1 (K <= 2 * kRowThreads).
  const float xmax = kk > 0 ? key_value(S.top[0]) : 0.f;
  float e[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int i = 2 * tid + q;
    e[q] = i < kk ? ex2(scaled(key_value(S.top[i]) - xmax, a.c_hi, a.c_lo)) : 0.f;
  }
  float sk;
  const float before = row_block_scan_f(e[0] + e[1], S, &sk);
  const float incl[2] = {before + e[0], before + e[0] + e[1]};
  const float norm = sk;  // the top-p mass is over the top K
  if (tid == 0) S.m = K;
  __syncthreads();
  if (a.top_p < 1.f) {
#pragma unroll
    for (int q = 1; q >= 0; --q)
      if (e[q] > 0.f && incl[q] / norm >= a.top_p) atomicMin(&S.m, 2 * tid + q + 1);
  }
  // min_p after top-p: the entries are in decreasing order, so it keeps the
  // prefix of those with 2^(c(x - xmax)) >= min_p.
  if (a.min_p > 0.f) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int i = 2 * tid + q;
      if (i < kk && e[q] < a.min_p) atomicMin(&S.m, i);
    }
  }
  __syncthreads();
  const int m = S.m;  // kept: the first m entries (zero weights past kk)
  if (2 * tid == m - 1) S.sm = incl[0];
  if (2 * tid + 1 == m - 1) S.sm = incl[1];
  __syncthreads();
  const float sm = S.sm;
  unsigned long long* rw = row_words_of(a, b, r);
  const int pos_x = r <= k ? r : r - k - 1;  // the draft token this row tests
  const int x = pos_x < kb ? a.tokens[(size_t)b * k + pos_x] : -1;
  float* pq = a.ws.pq + (size_t)b * 2 * k;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int i = 2 * tid + q;
    if (i < K) {
      const bool kept = i < kk && i < m && e[q] > 0.f;
      const float prob = kept ? e[q] / sm : 0.f;
      const int t = kept ? key_token(S.top[i]) : -1;
      rw[i] = kept ? ((unsigned long long)(t + 1) << 32) | __float_as_uint(prob) : 0ull;
      if (kept && t == x) pq[(r <= k ? 0 : k) + pos_x] = prob;
    }
  }
}

// The request's ticket (acquire-release: the row's published words before
// it, the other rows' after it); the last of its row CTAs finishes it.
__device__ __forceinline__ void row_done(RowSmem& S, const ChainArgs& a, int b) {
  const int R = 2 * a.k + 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                 : "=r"(t)
                 : "l"(&a.ws.sync[b].tick2)
                 : "memory");
    S.last = t == R - 1;
    if (S.last) {
      a.ws.sync[b].tick2 = 0;
      S.failed = atomicExch(&a.ws.sync[b].failed, 0);
    }
  }
  __syncthreads();
  if (S.last) finish_request(S, a, b);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kRowThreads, kRowCtasPerSm) filter_row_kernel(const __grid_constant__ ChainArgs a) {
  using IO = Io<DT, VEC>;
  constexpr int NW = IO::NW;
  __shared__ RowSmem S;
  const int tid = threadIdx.x;
  const int K = a.top_k, k = a.k, R = 2 * k + 1;
  const int b = blockIdx.x / R, r = blockIdx.x - b * R;
  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const int kb = (kraw < 0 || kraw > k) ? 0 : kraw;

  if (row_used(k, kraw, r)) {
    const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
    const int nvec = a.nvec;
    const int nch = ceil_div(nvec, kChunkVecs);
    if (tid == 0) {
      S.n = 0;
      S.kappa = 0;
      S.tcode = ~0u;
    }
    uint32_t X0[kRowVecs][NW], X1[kRowVecs][NW];
    load_chunk<DT, VEC>(row, 0, nvec, X0);
    if (nch > 1) load_chunk<DT, VEC>(row, 1, nvec, X1);
    __syncthreads();
    for (int c = 0; c < nch; c += 2) {  // chunk c + 2 loads while c + 1 is filtered
      filter_chunk<DT, VEC>(S, K, c, nvec, X0);
      if (c + 2 < nch) load_chunk<DT, VEC>(row, c + 2, nvec, X0);
      if (c + 1 < nch) {
        filter_chunk<DT, VEC>(S, K, c + 1, nvec, X1);
        if (c + 3 < nch) load_chunk<DT, VEC>(row, c + 3, nvec, X1);
      }
    }
    __syncthreads();
    publish_row(S, a, b, r, kb);
  }
  row_done(S, a, b);
}

// ------------------------------------------------------------------ rows with 16-byte vectors
// Pass 1, filter_max_kernel: one CTA per 32 KB slice of a row (request-major
// order), each thread's 8 vectors read once with 128-bit loads.  For each
// group of 8 contiguous vectors (128 bytes) it writes only the 16-bit prefix
// of the order bits of the group's largest logit (0: no finite logit), so
// the pass has the streaming shape of the unfiltered pass 1 without its
// exponentials.
// Pass 2, filter_pick_kernel: one CTA per row.  tau: a prefix that at
// least K of the row's group prefixes reach (per-warp bisections); at least
// K logits are >= tau (those groups' maxima), so the row's top K all lie in
// the groups whose prefix is >= tau (somewhat more than K of them).  Only
// those groups are read again (one 128-byte line each); their logits with
// key >= tau << 48 are the candidates.
constexpr int kSegSlices = 8;                     // slices per selection segment
constexpr int kPickVecs = 6;                      // vectors a pick thread reads per round
constexpr int kPickCtasPerSm = 7;                 // 1064 rows resident on 152 SMs
constexpr int kSegPairs = kSegSlices * kThreads;  // (slice, group) pairs per segment
constexpr int kMaxCodes = 56 * kThreads;          // codes a pick CTA holds (56 slices)
constexpr int kStage = 32;                        // vectors a pick warp packs per pass
constexpr int kSegReads = kSegPairs / 8 / kRowThreads;  // 16-byte code reads per thread
static_assert(kSegReads * 8 * kRowThreads == kSegPairs, "a segment's codes in 16-byte reads");
// The pick's static shared memory plus its codes stay within the 48 KB a
// launch may take without opting in to more.
static_assert(sizeof(RowSmem) + sizeof(unsigned short) * kSegPairs + sizeof(int) * kRowWarps * kStage +
                      sizeof(unsigned short) * kMaxCodes <= 48 * 1024,
              "filter_pick_kernel's shared memory");
static_assert(kRowWarps * kStage * 16 <= sizeof(unsigned long long) * SPEC_MAX_TOPK,
              "the pick's stage lives in RowSmem::top");

__device__ __forceinline__ uint4 ld_volatile_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.volatile.global.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
// Whether every 16-bit half of the eight codes is nonzero.
__device__ __forceinline__ bool all_halves_set(const uint4& v) {
  return __vcmpeq2(v.x, 0) == 0 && __vcmpeq2(v.y, 0) == 0 && __vcmpeq2(v.z, 0) == 0 &&
         __vcmpeq2(v.w, 0) == 0;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 6) filter_max_kernel(const ChainArgs a) {
  using IO = Io<DT, VEC>;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched by launch_first
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  const int rr = blockIdx.x / a.nsplit, s = blockIdx.x - rr * a.nsplit;
  const int R = 2 * a.k + 1;
  const int b = rr / R, r = rr - b * R;
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  const int vbeg = s * a.vps;
  // this thread's vectors vbeg + tid + u * kThreads, u < nv
  const int nv = min(kVecPerThread, max(0, min(a.nvec - vbeg, a.vps) - tid + kThreads - 1) / kThreads);
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES) + (size_t)(vbeg + tid) * (VEC ? 16 : IO::ES);
  uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u)
    if (u < nv) IO::load(row, u * kThreads, w[u]);
  // Group g of the slice = its vectors 8g .. 8g + 7 (128 contiguous bytes),
  // held by lanes 8 (g mod 4) .. + 7 of warp (g / 4) mod 8 for u = g / 32:
  // each lane's vector maximum, then the maximum over its eight lanes.
  unsigned short* out = a.ws.codes + (size_t)blockIdx.x * kThreads;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    float m = u < nv ? IO::vmax(w[u]) : -INFINITY;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // stored plus one: a written code is never 0 (the pick polls for it)
    if ((tid & 7) == 0) {
      const unsigned short c = (unsigned short)(m > -INFINITY ? (ord32(m) >> 16) + 1 : 1u);
      asm volatile("st.relaxed.gpu.global.u16 [%0], %1;" ::"l"(out + tid / 8 + u * (kThreads / 8)),
                   "h"(c)
                   : "memory");
    }
  }
}

// A threshold t with at least K of the n codes >= t (0 excluded; 0 when a
// warp holds fewer than cw nonzero codes): warp w takes codes w*32 + lane +
// 128 j and finds its cw-th largest (cw = ceil(K / 4); bisection between its
// least and largest nonzero code, ballot counts); t is the least of the four
// (no shared-memory atomics: the codes of a row cluster on few values).
__device__ uint32_t code_threshold(const unsigned short* codes, int n, int K, RowSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cw = (K + kRowWarps - 1) / kRowWarps;
  constexpr int kReg = kSegPairs / kRowThreads;  // codes per lane held in registers
  uint32_t c[kReg];
  const bool in_regs = n <= kSegPairs;
  uint32_t lo = ~0u, hi = 0;
  int nz = 0;
  if (in_regs) {
#pragma unroll
    for (int q = 0; q < kReg; ++q) {
      const int i = warp * 32 + lane + q * kRowThreads;
      c[q] = i < n ? codes[i] : 0u;
      if (c[q]) {
        lo = min(lo, c[q]);
        hi = max(hi, c[q]);
        ++nz;
      }
    }
  } else {
    for (int i = warp * 32 + lane; i < n; i += kRowThreads) {
      const uint32_t v = codes[i];
      if (v) {
        lo = min(lo, v);
        hi = max(hi, v);
        ++nz;
      }
    }
  }
  uint32_t t = 0;
  bool done = false;
  if (in_regs && cw <= 16) {
    // The cw-th largest of the lanes' two largest codes: those are distinct
    // codes of the warp, so at least cw codes reach it; it is below the
    // exact cw-th largest code only when a lane holds three or more of the
    // warp's top cw codes.  Two values per lane make the bisection cheap.
    uint32_t m1 = 0, m2 = 0;
#pragma unroll
    for (int q = 0; q < kReg; ++q) {
      m2 = max(m2, min(m1, c[q]));
      m1 = max(m1, c[q]);
    }
    const int nz2 = (int)__reduce_add_sync(0xffffffffu, (m1 != 0u ? 1u : 0u) + (m2 != 0u ? 1u : 0u));
    if (nz2 >= cw) {  // else the exact search below (e.g. a mostly masked vocabulary)
      uint32_t l2 = __reduce_min_sync(0xffffffffu, m2 != 0u ? m2 : (m1 != 0u ? m1 : ~0u));
      uint32_t h2 = __reduce_max_sync(0xffffffffu, m1);
      while (l2 < h2) {  // count(>= l2) >= cw over the 2 x 32 values
        const uint32_t mid = (l2 + h2 + 1) >> 1;
        const unsigned m = (m1 >= mid ? 1u : 0u) + (m2 >= mid ? 1u : 0u);
        if ((int)__reduce_add_sync(0xffffffffu, m) >= cw) l2 = mid;
        else h2 = mid - 1;
      }
      t = l2;
      done = true;
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  nz = (int)__reduce_add_sync(0xffffffffu, (unsigned)nz);
  if (!done && nz >= cw) {
    while (lo < hi) {  // the warp's nz >= cw codes are all >= lo
      const uint32_t mid = (lo + hi + 1) >> 1;
      unsigned m = 0;
      if (in_regs) {
#pragma unroll
        for (int q = 0; q < kReg; ++q) m += c[q] >= mid ? 1u : 0u;
      } else {
        for (int i = warp * 32 + lane; i < n; i += kRowThreads) m += codes[i] >= mid ? 1u : 0u;
      }
      if ((int)__reduce_add_sync(0xffffffffu, m) >= cw) lo = mid;
      else hi = mid - 1;
    }
    t = lo;
  }
  if (threadIdx.x == 0) S.tcode = ~0u;
  __syncthreads();
  if (lane == 0) atomicMin(&S.tcode, t);
  __syncthreads();
  t = S.tcode;
  __syncthreads();  // S.tcode is rewritten next
  return t;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kRowThreads, kPickCtasPerSm) filter_pick_kernel(
    const __grid_constant__ ChainArgs a) {
  using IO = Io<DT, VEC>;
  constexpr int NW = IO::NW;
  __shared__ RowSmem S;
  __shared__ unsigned short pairs[kSegPairs];  // (slice - segment start) << 8 | group
  __shared__ int stage_idx[kRowWarps * kStage];  // vector indices of the stage
  extern __shared__ unsigned short codes[];    // the row's thread prefixes
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.top_k, k = a.k, R = 2 * k + 1, ns = a.nsplit;
  const int b = blockIdx.x / R, r = blockIdx.x - b * R;
  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const int kb = (kraw < 0 || kraw > k) ? 0 : kraw;

  if (row_used(k, kraw, r)) {
    const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
    const int n = ns * kThreads;
    // The row's codes as pass 1 writes them (eight per 16-byte load; a
    // 16-bit half still 0 is not written yet: wait for it, bounded), stored
    // back decoded (0 = no finite logit).
    uint4* g = reinterpret_cast<uint4*>(a.ws.codes + (size_t)blockIdx.x * n);
    bool to = false;  // a wait of this thread ran out
    for (int i = tid; i < n / 8; i += kRowThreads) {
      uint4 v = ld_volatile_v4(g + i);
      const long long t0 = clock64();
      while (!all_halves_set(v)) {
        if (clock64() - t0 > a.wait_cycles) {
          set_status(a.ws.status, SPEC_ETIMEOUT);
          to = true;
          break;
        }
        __nanosleep(256);
        v = ld_volatile_v4(g + i);
      }
      // minus one per half (a half still 0 after a timeout stays 0)
      const uint32_t m1[4] = {v.x, v.y, v.z, v.w};
      uint32_t d[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) d[q] = __vsubus2(m1[q], 0x00010001u);
      reinterpret_cast<uint4*>(codes)[i] = make_uint4(d[0], d[1], d[2], d[3]);
      g[i] = make_uint4(0, 0, 0, 0);  // every call leaves the workspace zero
    }
    // A code or statistics word that never arrived: the request fails closed
    // (the flag reaches the finishing row CTA through the acquire-release
    // ticket).
    if (__syncthreads_or(to) && tid == 0) atomicExch(&a.ws.sync[b].failed, 1);
    if (tid == 0) S.n = 0;
    __syncthreads();
    const uint32_t tau = code_threshold(codes, n, K, S);
    if (tid == 0) {
      S.kappa = (unsigned long long)tau << 48;
      S.tcode = ~0u;  // for raise_held
    }
    __syncthreads();
    // The groups whose prefix is >= tau, a segment of slices at a time;
    // their vectors, kPickVecs per CTA thread per round.
    for (int s0 = 0; s0 < ns; s0 += kSegSlices) {
      const int s1 = min(ns, s0 + kSegSlices);
      // The segment's codes, eight per 16-byte read (kSegReads per thread):
      // an 8-bit mask of those >= max(tau, 1) each; a pair is the code's
      // index within the segment, ((s - s0) << 8) | group.
      const int c0 = s0 * kThreads, nseg = (s1 - s0) * kThreads;
      const uint32_t th = max(tau, 1u), th2 = th | (th << 16);
      uint32_t mk[kSegReads];
      int mine = 0;
#pragma unroll
      for (int h = 0; h < kSegReads; ++h) {
        const int v = tid + h * kRowThreads;  // codes 8v .. 8v + 7 of the segment
        mk[h] = 0;
        if (8 * v < nseg) {
          const uint4 x = reinterpret_cast<const uint4*>(codes + c0)[v];
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t ge = __vcmpgeu2(w[q], th2);  // 0xffff per half >= th
            mk[h] |= ((ge & 1u) | ((ge >> 15) & 2u)) << (2 * q);
          }
        }
        mine += __popc(mk[h]);
      }
      int npairs;
      int off = row_block_scan(mine, S, &npairs);
#pragma unroll
      for (int h = 0; h < kSegReads; ++h)
        for (uint32_t m = mk[h]; m; m &= m - 1)
          pairs[off++] = (unsigned short)(8 * (tid + h * kRowThreads) + __ffs(m) - 1);
      __syncthreads();
      const int items = npairs * kVecPerThread;  // (pair, vector) items
      for (int i0 = 0; i0 < items; i0 += kRowThreads * kPickVecs) {
        uint32_t X[kPickVecs][NW];
        int vidx[kPickVecs];
        float vm[kPickVecs];
#pragma unroll
        for (int u = 0; u < kPickVecs; ++u) {
          const int i = i0 + tid + u * kRowThreads;
          vidx[u] = -1;
          if (i < items) {
            const int p = pairs[i / kVecPerThread], uu = i % kVecPerThread;
            const int s = s0 + (p >> 8), g = p & 0xff;
            const int vbeg = s * a.vps, nvs = min(a.nvec, vbeg + a.vps) - vbeg;
            if (8 * g + uu < nvs) {
              vidx[u] = vbeg + 8 * g + uu;
              IO::load(row, vidx[u], X[u]);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kPickVecs; ++u) vm[u] = vidx[u] >= 0 ? IO::vmax(X[u]) : -INFINITY;
        // Of a selected group's eight vectors usually one reaches kappa, and
        // its eight lanes sit side by side in a warp: filtered in place, most
        // lanes would idle through every vector.  So the warp first packs the
        // vectors that can hold a candidate (maximum >= kappa) into its stage,
        // kStage at a time, and each lane then filters one of them.
        const float kv0 = S.kappa ? key_value(S.kappa) : -INFINITY;
        bool pass[kPickVecs];
        int mine = 0;
#pragma unroll
        for (int u = 0; u < kPickVecs; ++u) {
          pass[u] = vidx[u] >= 0 && vm[u] >= kv0 && vm[u] > -INFINITY;
          mine += pass[u] ? 1 : 0;
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int wtot = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t* stx = reinterpret_cast<uint32_t*>(S.top) + warp * kStage * NW;
        int* sti = stage_idx + warp * kStage;
        for (int b0 = 0; __syncthreads_or(b0 < wtot); b0 += kStage) {
          int sl = incl - mine - b0;
#pragma unroll
          for (int u = 0; u < kPickVecs; ++u)
            if (pass[u]) {
              if (sl >= 0 && sl < kStage) {
#pragma unroll
                for (int w = 0; w < NW; ++w) stx[sl * NW + w] = X[u][w];
                sti[sl] = vidx[u];
              }
              ++sl;
            }
          __syncwarp();
          uint32_t Y[1][NW];
          int yidx[1] = {-1};
          float ym[1] = {-INFINITY};
          if (b0 + lane < wtot) {
#pragma unroll
            for (int w = 0; w < NW; ++w) Y[0][w] = stx[lane * NW + w];
            yidx[0] = sti[lane];
            ym[0] = IO::vmax(Y[0]);
          }
          const unsigned long long kap = S.kappa;  // raised by an earlier pass, perhaps
          const float kv = kap ? key_value(kap) : -INFINITY;
          int cnt = 0;
          if (ym[0] >= kv && ym[0] > -INFINITY)
            vec_candidates<DT, VEC>(yidx[0], Y[0], kap, [&](unsigned long long) { ++cnt; });
          // (the stage is read before this barrier and rewritten only after
          // the next one; a cut inside may use S.top as scratch meanwhile)
          if (__syncthreads_or(cnt > 0)) append_chunk<DT, VEC, 1>(S, K, yidx, Y, ym, cnt);
        }
      }
      __syncthreads();  // pairs is rewritten by the next segment
    }
    __syncthreads();
    publish_row(S, a, b, r, kb);
  }
  row_done(S, a, b);
  // Completion of this grid then implies completion of pass 1.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

constexpr int kHash = 2 * SPEC_MAX_TOPK;       // slots of the finisher's token table
constexpr int kDrawBits = 9;                   // 2^9 token buckets per level of the draw search
constexpr int kDrawBuckets = 1 << kDrawBits;
constexpr int kDrawPerLane = kDrawBuckets / 32;
static_assert((kHash & (kHash - 1)) == 0 && kHash / 2 + kHash / 2 + SPEC_MAX_TOPK <= kBufCap,
              "the finisher's tables live in RowSmem::buf");
static_assert(kDrawBuckets <= kHash, "the draw's buckets reuse the token table");

// Slot of a token in the finisher's table: the top bits of a multiplicative
// (Fibonacci) hash.
__device__ __forceinline__ uint32_t hash_slot(uint32_t t) {
  return (t * 2654435761u) >> (32 - 9);
}
static_assert(kHash == 1 << 9, "hash_slot yields 9 bits");

// Exact warp-wide sum of 64-bit values whose total is below 2^64: three
// 21/22-bit pieces summed with 32-bit reductions.
__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long s) {
  const unsigned p0 = __reduce_add_sync(0xffffffffu, (unsigned)(s & 0x1fffffu));
  const unsigned p1 = __reduce_add_sync(0xffffffffu, (unsigned)((s >> 21) & 0x1fffffu));
  const unsigned p2 = __reduce_add_sync(0xffffffffu, (unsigned)(s >> 42));
  return ((unsigned long long)p2 << 42) + ((unsigned long long)p1 << 21) + p0;
}

// The request's last row CTA finishes it: accept scan, final draw, outputs,
// cleanup (thread t: position t of the scan; entries t and t + kRowThreads
// of target and draft row j's kept lists; warp 0 runs the draw's search).
__device__ __noinline__ void finish_request(RowSmem& S, const ChainArgs& a, int b) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, R = 2 * k + 1, K = a.top_k;
  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const bool bad_len = kraw < 0 || kraw > k;
  const int kb = bad_len ? 0 : kraw;
  float* pq = a.ws.pq + (size_t)b * 2 * k;
  float P = 0.f, Q = 0.f, U = 0.f;
  bool bad = bad_len;
  int x = -1;  // draft token tid
  if (tid < kb) {
    x = a.tokens[(size_t)b * k + tid];
    bad = x < 0 || x >= a.V;
    P = __ldcg(pq + tid);
    Q = __ldcg(pq + k + tid);
  }
  if (tid <= k)
    U = a.uniforms ? a.uniforms[(size_t)b * (k + 1) + tid]
                   : philox_uniform(a.seeds[b], a.offsets[b], tid);
  if (tid == 0) S.m = kb;
  if (tid == kb) S.sm = U;  // the final draw's uniform
  const bool any_bad = __syncthreads_or(bad);
  // accept x_i iff r_i < p_i(x_i) / q_i(x_i) (q = 0 accepts); j = the first rejection
  const float ratio = Q > 0.f ? P / Q : INFINITY;
  if (tid < kb && !(U < ratio)) atomicMin(&S.m, tid);
  __syncthreads();
  const int j = (any_bad || S.failed) ? -1 : S.m;
  const double u = (double)S.sm;
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (j >= 0) {
    // Target row j's kept list (token, p) and, when j < kb, draft row j's:
    // the latter goes into a hash table keyed by token (open addressing,
    // at most SPEC_MAX_TOPK keys in kHash slots), so q_j of each target
    // token is one or two probes.  The draw weights max(0, p - q_j) (bonus
    // row: p) are exact 64-bit fixed point (to_fixed of a value scaled by
    // 2^31, each < 2^32 before scaling).
    uint32_t* hk = reinterpret_cast<uint32_t*>(S.buf);                  // token + 1; 0 = empty
    float* hv = reinterpret_cast<float*>(S.buf + kHash / 2);            // its q
    int* T = reinterpret_cast<int*>(S.buf + kHash);                     // kept tokens
    float* Pj = reinterpret_cast<float*>(S.buf + kHash + SPEC_MAX_TOPK / 2);  // their p
    unsigned long long* F = S.top;                                      // draw weights
    unsigned long long wt[2], wd[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = tid + h * kRowThreads;
      wt[h] = i < K ? __ldcg(row_words_of(a, b, j) + i) : 0ull;
      wd[h] = (j < kb && i < K) ? __ldcg(row_words_of(a, b, k + 1 + j) + i) : 0ull;
    }
    for (int i = tid; i < kHash; i += kRowThreads) hk[i] = 0u;
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (wd[h]) {  // tokens of one kept list are distinct: each finds a free slot
        const uint32_t key = (uint32_t)(wd[h] >> 32);
        uint32_t slot = hash_slot(key - 1);
        for (int probe = 0; probe < kHash; ++probe, slot = (slot + 1) & (kHash - 1))
          if (atomicCAS(&hk[slot], 0u, key) == 0u) {
            hv[slot] = __uint_as_float((uint32_t)wd[h]);
            break;
          }
      }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = tid + h * kRowThreads;
      if (i < K) {
        const int tk = wt[h] ? (int)(wt[h] >> 32) - 1 : INT_MAX;
        const float p = wt[h] ? __uint_as_float((uint32_t)wt[h]) : 0.f;
        float qv = 0.f;
        if (wt[h] && j < kb) {
          uint32_t slot = hash_slot((uint32_t)tk);
          for (int probe = 0; probe < kHash; ++probe, slot = (slot + 1) & (kHash - 1)) {
            const uint32_t key = hk[slot];
            if (key == (uint32_t)tk + 1u) {
              qv = hv[slot];
              break;
            }
            if (key == 0u) break;
          }
        }
        F[i] = wt[h] ? to_fixed(fmaxf(p - qv, 0.f) * 2147483648.0f) : 0ull;
        T[i] = tk;
        Pj[i] = p;
      }
    }
    __syncthreads();
    // Inverse CDF in token order without sorting, in warp 0: Z = the sum of
    // the weights, target = floor(u Z) < Z, and the drawn token is the least
    // t whose cumulative weight over kept tokens <= t exceeds target; that
    // token has nonzero weight and the weights of the kept tokens below it
    // sum to at most target.  Search: the token range [lo, hi] is split into
    // at most kDrawBuckets buckets of 2^sh tokens whose weights are summed
    // exactly (64-bit shared atomics); the bucket holding target (lane-local
    // then warp scans) becomes the range, until one token is left (two
    // levels for V <= 2^18).  Lane l owns buckets 16 l .. 16 l + 15, stored
    // transposed (bucket b at (b mod 16) * 32 + b / 16).
    if (warp == 0) {
      unsigned long long sum = 0;
      for (int i = lane; i < K; i += 32) sum += F[i];
      unsigned long long Z = warp_sum_u64(sum);
      if (Z == 0) {  // the residual vanished numerically: draw from p_j
        sum = 0;
        for (int i = lane; i < K; i += 32) {
          F[i] = T[i] != INT_MAX ? to_fixed(Pj[i] * 2147483648.0f) : 0ull;
          sum += F[i];
        }
        Z = warp_sum_u64(sum);
        __syncwarp();
      }
      int lo = 0;  // no kept token at all (a row without a finite logit): token 0
      if (Z != 0) {
        unsigned long long target = (unsigned long long)(u * (double)Z);  // < Z
        unsigned long long* bk = S.buf;  // the token table is done with
        int hi = a.V - 1;                // weight in [lo, hi] = Z > target
        while (lo < hi) {
          // 2^sh tokens per bucket, sh the least with kDrawBuckets << sh > hi - lo
          const int sh = max(0, 32 - __clz(hi - lo) - kDrawBits);
#pragma unroll
          for (int q = 0; q < kDrawPerLane; ++q) bk[q * 32 + lane] = 0ull;
          __syncwarp();
          for (int i = lane; i < K; i += 32) {
            const unsigned long long fi = F[i];
            const int ti = T[i];
            if (fi != 0ull && ti >= lo && ti <= hi) {
              const int bb = (ti - lo) >> sh;
              atomicAdd(&bk[(bb % kDrawPerLane) * 32 + bb / kDrawPerLane], fi);
            }
          }
          __syncwarp();
          unsigned long long own = 0;  // the lane's buckets in all
#pragma unroll
          for (int q = 0; q < kDrawPerLane; ++q) own += bk[q * 32 + lane];
          unsigned long long incl = own;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
          }
          const unsigned long long ex = incl - own;
          const unsigned hit = __ballot_sync(0xffffffffu, ex <= target && target < incl);
          const int src = __ffs(hit) - 1;
          // in the lane that holds target: its bucket (the buckets wholly
          // below target are those whose inclusive sum is <= target - ex)
          // and the weight below it
          int idx = 0;
          unsigned long long below = 0, run = 0;
#pragma unroll
          for (int q = 0; q < kDrawPerLane; ++q) {
            run += bk[q * 32 + lane];
            if (run <= target - ex) {
              ++idx;
              below = run;
            }
          }
          const int bucket = __shfl_sync(0xffffffffu, lane * kDrawPerLane + idx, src);
          target -= __shfl_sync(0xffffffffu, ex + below, src);
          __syncwarp();  // the buckets are cleared next
          lo += bucket << sh;
          hi = min(hi, lo + (1 << sh) - 1);
        }
      }
      if (lane == 0) S.red = lo;
    }
    __syncthreads();
    const int drawn = S.red;
    for (int i = tid; i <= k; i += kRowThreads)  // (i < j <= kb: thread i holds x_i)
      out[i] = i < j ? (i == tid ? x : a.tokens[(size_t)b * k + i]) : (i == j ? drawn : -1);
    if (a.out_probs && tid < k) {  // padded positions are not verified: NaN
      a.out_probs[((size_t)b * k + tid) * 2] = tid < kb ? P : NAN;
      a.out_probs[((size_t)b * k + tid) * 2 + 1] = tid < kb ? Q : NAN;
    }
    if (tid == 0) {
      a.out_n[b] = j;
      if (a.seq_lens) a.seq_lens[b] += j + 1;
    }
  } else {  // a bad draft token or length, or a wait ran out: fail closed
    for (int i = tid; i <= k; i += kRowThreads) out[i] = -1;
    if (a.out_probs)
      for (int i = tid; i < 2 * k; i += kRowThreads) a.out_probs[(size_t)b * 2 * k + i] = NAN;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a.ws.status, SPEC_EBADINDEX);
    }
  }
  // Every call leaves the workspace zero: the kept lists and probabilities.
  for (int r = 0; r < R; ++r)
    if (row_used(k, kraw, r)) {
      unsigned long long* rw = row_words_of(a, b, r);
      for (int i = tid; i < K; i += kRowThreads) rw[i] = 0;
    }
  for (int i = tid; i < 2 * k; i += kRowThreads) pq[i] = 0.f;
}

template <int DT, bool VEC>
cudaError_t launch_filtered_t(const ChainArgs& a, cudaStream_t st, bool skip_pass1) {
  const long rows = (long)a.B * (2 * a.k + 1);
  if ((long)a.nsplit * kThreads <= kMaxCodes) {
    if (!skip_pass1) {
      const cudaError_t e = launch_first(filter_max_kernel<DT, VEC>, rows * a.nsplit, kThreads, st, a);
      if (e != cudaSuccess) return e;
    }
    // The pick grid may be scheduled once every pass-1 CTA has started; each
    // row CTA waits only for its own row's codes.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = sizeof(unsigned short) * a.nsplit * kThreads;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, filter_pick_kernel<DT, VEC>, a);
  } else {  // a row too wide for one CTA's prefixes: stream it through one CTA
    if (skip_pass1) return cudaErrorNotSupported;  // one pass: nothing to wait for
    filter_row_kernel<DT, VEC><<<(unsigned)rows, kRowThreads, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_filtered(const ChainArgs& a, int dtype, bool vec, cudaStream_t st,
                            bool skip_pass1) {
  if (dtype == SPEC_BF16)
    return vec ? launch_filtered_t<SPEC_BF16, true>(a, st, skip_pass1)
               : launch_filtered_t<SPEC_BF16, false>(a, st, skip_pass1);
  return vec ? launch_filtered_t<SPEC_F32, true>(a, st, skip_pass1)
             : launch_filtered_t<SPEC_F32, false>(a, st, skip_pass1);
}

}  // namespace sv
