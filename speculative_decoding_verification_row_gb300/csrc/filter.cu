// Chain rejection-sampling verify on top-k / top-p filtered distributions
// (TensorRT-LLM walkthrough, rejection-sampling section: the target side is
// filtered by the same backend and parameters as the draft side was, or the
// accept test is silently wrong).  Every target and draft row is reduced to
// its kept set: the top_k tokens by (logit descending, token ascending), then
// the shortest prefix of them whose softmax mass (softmax over those top_k,
// at temperature T) reaches top_p; p and q are the softmax over the kept set.
// The verify itself is the plain chain rule (vLLM anatomy page, "Speculative
// Decoding"): accept x_i iff r_i < p_i(x_i) / q_i(x_i) (q = 0 accepts), stop
// at the first rejection j and draw from max(0, p_j - q_j) normalised, or
// from p_k when all k are accepted.
//
// Since p_j is zero outside target row j's kept set, the final draw has at
// most top_k candidate tokens, so after one streaming pass nothing re-reads a
// logit row.
//
// Pass 1, filter_topk_kernel: one CTA per 32 KB slice of a row (request-major
// order, as the unfiltered pass 1).  It publishes the slice's top_k keys,
// sorted, as nonzero 64-bit words.  A key is (order-preserving bits of the
// logit) << 32 | (2^32 - 1 - token): larger key = larger logit, then lower
// token.  Logits of -inf are never kept: their weight is exactly 0, so they
// change no probability, no top-p prefix and no draw.
//   Selection: each thread's largest logit; a bisection over the 256 thread
//   maxima (one block-wide count per bit) finds tau, the top_k-th largest of
//   them.  At least top_k elements are >= tau, so the slice's top_k all are:
//   the vectors holding an element >= tau (about top_k of 2048) are copied
//   to shared memory, their elements >= tau become keys, and a bitonic sort
//   orders them.  When those do not fit (many equal logits), an exact
//   bisection over the elements' values, then over the tied tokens' indices,
//   selects exactly the top_k.
// Pass 2, filter_finish_kernel: a programmatic dependent of pass 1; one CTA
// item per (request, row).  It polls the row's slice lists, merges them by
// rank (a key's rank is its position in its own list plus the keys above it
// in each other list, found by binary search), applies the softmax and the
// top-p cut to the top_k, and writes the row's kept list (token, probability)
// and, for the rows that test a draft token, that token's probability.  The
// request's last row item (atomic ticket) runs the accept scan and draws the
// final token by inverse CDF over the kept tokens of target row j in token
// order, with exact 64-bit fixed-point prefix sums.
#include <mutex>

#include "kernels.cuh"

namespace sv {

namespace {

constexpr unsigned long long kNone = 1;  // an empty slot: below every real key
constexpr int kQCap = 512;               // candidate vectors one slice CTA holds
constexpr int kCCap = 1024;              // candidate keys one slice CTA sorts

// Order-preserving map of a float (not NaN) to 32 bits, -0 taken as +0.
__device__ __forceinline__ uint32_t ord32(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord32(uint32_t o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}
__device__ __forceinline__ unsigned long long make_key(float x, long t) {
  return ((unsigned long long)ord32(x) << 32) | (0xffffffffu - (uint32_t)t);
}
__device__ __forceinline__ float key_value(unsigned long long key) {
  return unord32((uint32_t)(key >> 32));
}
__device__ __forceinline__ int key_token(unsigned long long key) {
  return (int)(0xffffffffu - (uint32_t)key);
}

// Block-wide sum of one int per thread (all threads call; every thread gets it).
__device__ __forceinline__ int block_sum(int v, int* scratch) {
  const int w = __reduce_add_sync(0xffffffffu, (unsigned)v);
  __syncthreads();  // earlier readers of *scratch are done
  if (threadIdx.x == 0) *scratch = 0;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) atomicAdd(scratch, w);
  __syncthreads();
  return *scratch;
}

// Bitonic sort of n 64-bit keys in shared memory, descending (ascending when
// ASC), padded with `pad` to a power of two; returns the padded length.
template <bool ASC>
__device__ int bitonic_sort(unsigned long long* keys, int n, unsigned long long pad) {
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = n + threadIdx.x; i < P; i += blockDim.x) keys[i] = pad;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
        const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
        const bool first_half_down = ((lo & size) == 0) != ASC;  // this block's direction
        const unsigned long long x = keys[lo], y = keys[hi];
        if ((x < y) == first_half_down) {
          keys[lo] = y;
          keys[hi] = x;
        }
      }
    }
  }
  __syncthreads();
  return P;
}

// Number of keys above `key` in a descending list of n keys.
__device__ __forceinline__ int count_above(const unsigned long long* list, int n,
                                           unsigned long long key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (list[mid] > key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Inclusive prefix sum across the block (fp32 or u64); *total gets the sum.
template <typename T>
__device__ __forceinline__ T block_incl_scan(T v, T* warp_tot, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  __syncthreads();  // earlier readers of warp_tot are done
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  T base = T(0), all = T(0);
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const T t = warp_tot[w];
    if (w < warp) base += t;
    all += t;
  }
  *total = all;
  return base + v;
}

__device__ __forceinline__ void slice_row(const ChainArgs& a, int rr, int& b, int& r) {
  const int R = 2 * a.k + 1;
  b = rr / R;
  r = rr - b * R;
}

// ------------------------------------------------------------------ pass 1
template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) filter_topk_kernel(const ChainArgs a) {
  asm volatile("griddepcontrol.launch_dependents;");
  using IO = Io<DT, VEC>;
  constexpr int EPV = IO::EPV, NW = IO::NW;
  // bf16 logits widened to fp32 differ only in their top 16 bits.
  constexpr int LOBIT = DT == SPEC_BF16 ? 16 : 0;
  __shared__ uint32_t sVec[kQCap][NW];
  __shared__ int sVecIdx[kQCap];
  __shared__ unsigned long long sKey[kCCap];
  __shared__ int sNV, sNC, sCnt;
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = a.top_k;
  const int rr = blockIdx.x / a.nsplit, s = blockIdx.x - rr * a.nsplit;
  int b, r;
  slice_row(a, rr, b, r);
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
  const int vbeg = s * a.vps;
  const int vend = min(a.nvec, vbeg + a.vps);

  uint32_t w[kVecPerThread][NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + tid + u * kThreads;
    if (v < vend) IO::load(row, v, w[u]);
  }
  float vm[kVecPerThread];
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    vm[u] = vbeg + tid + u * kThreads < vend ? IO::vmax(w[u]) : -INFINITY;
    m = fmaxf(m, vm[u]);
  }
  if (tid == 0) {
    sNV = 0;
    sNC = 0;
  }
  // tau = the K-th largest thread maximum (0: fewer than K threads hold a
  // finite logit, and every finite logit is a candidate).
  const uint32_t mo = m > -INFINITY ? ord32(m) : 0u;
  uint32_t t = 0;
  for (int bit = 31; bit >= LOBIT; --bit) {
    const uint32_t c = t | (1u << bit);
    if (__syncthreads_count(mo >= c) >= K) t = c;
  }
  if (LOBIT && t && !(t & 0x80000000u)) t |= 0xffffu;  // the bf16 value's own code
  const float tau = t ? unord32(t) : -INFINITY;

  // Copy every vector holding a candidate (x >= tau, x > -inf) to shared memory.
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + tid + u * kThreads;
    const bool hit = v < vend && vm[u] >= tau && vm[u] > -INFINITY;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (bal) {
      int base = 0;
      if (lane == 0) base = atomicAdd(&sNV, __popc(bal));
      base = __shfl_sync(0xffffffffu, base, 0);
      const int slot = base + __popc(bal & ((1u << lane) - 1u));
      if (hit && slot < kQCap) {
#pragma unroll
        for (int q = 0; q < NW; ++q) sVec[slot][q] = w[u][q];
        sVecIdx[slot] = v;
      }
    }
  }
  __syncthreads();
  const int nv = sNV;
  if (nv <= kQCap) {
    for (int i = tid; i < nv; i += kThreads) {
      uint32_t ww[NW];
#pragma unroll
      for (int q = 0; q < NW; ++q) ww[q] = sVec[i][q];
      float e[EPV];
      IO::unpack(ww, e);
      const long t0 = (long)sVecIdx[i] * EPV;
#pragma unroll
      for (int q = 0; q < EPV; ++q)
        if (e[q] >= tau && e[q] > -INFINITY) {
          const int slot = atomicAdd(&sNC, 1);
          if (slot < kCCap) sKey[slot] = make_key(e[q], t0 + q);
        }
    }
  }
  __syncthreads();
  int nc = sNC;
  if (nv > kQCap || nc > kCCap) {
    // Exact selection (many equal logits).  First the K-th largest finite
    // value tv (bisection on its order bits), then, if the logits equal to tv
    // are too many to sort, the highest token index among them that is kept.
    auto count_if = [&](auto pred) {
      int c = 0;
#pragma unroll
      for (int u = 0; u < kVecPerThread; ++u) {
        const int v = vbeg + tid + u * kThreads;
        if (v < vend) {
          float e[EPV];
          IO::unpack(w[u], e);
#pragma unroll
          for (int q = 0; q < EPV; ++q) c += pred(e[q], (long)v * EPV + q) ? 1 : 0;
        }
      }
      return block_sum(c, &sCnt);
    };
    const int finite = count_if([](float x, long) { return x > -INFINITY; });
    float tv = -INFINITY;
    if (finite > K) {
      uint32_t o = 0;
      for (int bit = 31; bit >= LOBIT; --bit) {
        const uint32_t c = o | (1u << bit);
        if (count_if([&](float x, long) { return x > -INFINITY && ord32(x) >= c; }) >= K) o = c;
      }
      if (LOBIT && !(o & 0x80000000u)) o |= 0xffffu;  // the bf16 value's own code
      tv = unord32(o);
    }
    const int above = count_if([&](float x, long) { return x > -INFINITY && x > tv; });
    const int ties = count_if([&](float x, long) { return x > -INFINITY && x == tv; });
    long tmax = LONG_MAX;  // tied tokens above this index are not kept
    if (above + ties > kCCap) {
      const int need = K - above;  // 1 <= need <= ties
      long lo = (long)vbeg * EPV, hi = (long)vend * EPV - 1;
      while (lo < hi) {  // smallest index with `need` ties at or below it
        const long mid = lo + (hi - lo) / 2;
        if (count_if([&](float x, long tt) { return x > -INFINITY && x == tv && tt <= mid; }) >= need)
          hi = mid;
        else
          lo = mid + 1;
      }
      tmax = lo;
    }
    __syncthreads();
    if (tid == 0) sNC = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = vbeg + tid + u * kThreads;
      if (v < vend) {
        float e[EPV];
        IO::unpack(w[u], e);
#pragma unroll
        for (int q = 0; q < EPV; ++q) {
          const long tt = (long)v * EPV + q;
          if (e[q] > -INFINITY && (e[q] > tv || (e[q] == tv && tt <= tmax))) {
            const int slot = atomicAdd(&sNC, 1);
            if (slot < kCCap) sKey[slot] = make_key(e[q], tt);
          }
        }
      }
    }
    __syncthreads();
    nc = min(sNC, kCCap);
  }
  bitonic_sort<false>(sKey, nc, 0ull);
  unsigned long long* out =
      a.ws.cand + (((size_t)b * (2 * a.k + 1) + r) * a.nsplit + s) * (size_t)K;
  for (int i = tid; i < K; i += kThreads) st_relaxed_u64(out + i, i < nc ? sKey[i] : kNone);
}

// ------------------------------------------------------------------ pass 2
// One (request, row) item: merge, filter, publish; the request's last item
// finishes the request.
__device__ void filter_row_item(const ChainArgs& a, int b, int r, unsigned long long* sL) {
  __shared__ unsigned long long sTop[kThreads];
  __shared__ float sWarpF[kWarps];
  __shared__ unsigned long long sWarpU[kWarps];
  __shared__ float sP[SPEC_MAX_DRAFT], sQ[SPEC_MAX_DRAFT], sU[SPEC_MAX_DRAFT + 1];
  __shared__ int sM, sJ, sLast, sTok;
  __shared__ float sSm;
  const int tid = threadIdx.x;
  const int k = a.k, R = 2 * k + 1, K = a.top_k, ns = a.nsplit;
  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const bool bad_len = kraw < 0 || kraw > k;
  const int kb = bad_len ? 0 : kraw;
  auto row_words = [&](int rr) {
    return a.ws.cand + ((size_t)b * R + rr) * (size_t)ns * K;
  };
  float* pq = a.ws.pq + (size_t)b * 2 * k;

  if (row_used(k, kraw, r)) {
    unsigned long long* rw = row_words(r);
    const int n = ns * K;
    for (int i = tid; i < n; i += kThreads) {
      unsigned long long v = ld_relaxed_u64(rw + i);
      if (!v) v = wait_word(rw + i, a.ws.status, kNone);
      sL[i] = v;
    }
    if (tid < K) sTop[tid] = kNone;
    if (tid == 0) sM = K;
    __syncthreads();
    // Global rank of each key: its place in its own (descending) list plus
    // the keys above it in every other list (keys are unique).
    for (int i = tid; i < n; i += kThreads) {
      const unsigned long long key = sL[i];
      if (key == kNone) continue;
      const int sl = i / K;
      int rank = i - sl * K;
      for (int s2 = 0; s2 < ns && rank < K; ++s2)
        if (s2 != sl) rank += count_above(sL + (size_t)s2 * K, K, key);
      if (rank < K) sTop[rank] = key;
    }
    __syncthreads();
    for (int i = K + tid; i < n; i += kThreads) rw[i] = 0;  // the first K words get the kept list

    // Softmax over the top K (temperature T), then the top-p cut.
    const unsigned long long key = tid < K ? sTop[tid] : kNone;
    const bool real = key != kNone;
    const float xmax = sTop[0] != kNone ? key_value(sTop[0]) : 0.f;
    const float e = real ? ex2(scaled(key_value(key) - xmax, a.c_hi, a.c_lo)) : 0.f;
    float sk;
    const float incl = block_incl_scan(e, sWarpF, &sk);
    if (a.top_p < 1.f && real && incl / sk >= a.top_p) atomicMin(&sM, tid + 1);
    __syncthreads();
    const int m = sM;  // kept: the first m (ranks past the real keys carry no weight)
    if (tid == m - 1) sSm = incl;
    __syncthreads();
    const float prob = (real && tid < m) ? e / sSm : 0.f;
    const int tok = real ? key_token(key) : -1;
    if (tid < K)
      rw[tid] = (real && tid < m)
                    ? ((unsigned long long)(tok + 1) << 32) | __float_as_uint(prob)
                    : 0ull;
    // The probability of the draft token this row tests.
    const int pos = r <= k ? r : r - k - 1;
    if (pos < kb && tok >= 0 && tid < m) {
      const int x = a.tokens[(size_t)b * k + pos];
      if (x == tok) pq[(r <= k ? 0 : k) + pos] = prob;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int t = atomicAdd(&a.ws.sync[b].tick2, 1);
    sLast = t == R - 1;
    if (sLast) {
      a.ws.sync[b].tick2 = 0;
      __threadfence();
    }
  }
  __syncthreads();
  if (!sLast) return;

  // ---------------------------------------------------------- finish
  bool bad = bad_len;
  if (tid < kb) {
    const int x = a.tokens[(size_t)b * k + tid];
    bad = x < 0 || x >= a.V;
    sP[tid] = __ldcg(pq + tid);
    sQ[tid] = __ldcg(pq + k + tid);
  }
  if (tid <= k)
    sU[tid] = a.uniforms ? a.uniforms[(size_t)b * (k + 1) + tid]
                         : philox_uniform(a.seeds[b], a.offsets[b], tid);
  const int any_bad = __syncthreads_or(bad);
  if (tid < 32) {  // accept scan: r_i < p_i(x_i) / q_i(x_i), q == 0 accepts
    unsigned rej[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = tid + 32 * h;
      bool rj = false;
      if (i < kb) {
        const float ratio = sQ[i] > 0.f ? sP[i] / sQ[i] : INFINITY;
        rj = !(sU[i] < ratio);
      }
      rej[h] = __ballot_sync(0xffffffffu, rj);
    }
    if (tid == 0) sJ = any_bad ? -1 : rej[0] ? __ffs(rej[0]) - 1 : rej[1] ? 31 + __ffs(rej[1]) : kb;
  }
  __syncthreads();
  const int j = sJ;
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (j >= 0) {
    // Kept tokens of target row j in token order, with p and the weight
    // max(0, p - q_j) (bonus row: p).
    const unsigned long long* pw = row_words(j);
    unsigned long long* sQW = sL;  // draft row j's kept list
    if (j < kb)
      for (int i = tid; i < K; i += kThreads) sQW[i] = __ldcg(row_words(k + 1 + j) + i);
    const unsigned long long word = tid < K ? __ldcg(pw + tid) : 0ull;
    sTop[tid] = word ? word - (1ull << 32) : ~0ull;  // (token << 32 | p bits), ascending sort
    __syncthreads();
    bitonic_sort<true>(sTop, kThreads, ~0ull);
    const unsigned long long ent = sTop[tid];
    const bool kept = ent != ~0ull;
    const int tok = kept ? (int)(ent >> 32) : -1;
    const float p = kept ? __uint_as_float((uint32_t)ent) : 0.f;
    float q = 0.f;
    if (kept && j < kb)
      for (int i = 0; i < K; ++i) {
        const unsigned long long qe = sQW[i];
        if ((int)(qe >> 32) == tok + 1) {
          q = __uint_as_float((uint32_t)qe);
          break;
        }
      }
    // Exact prefix sums of the weights scaled by 2^31 (each < 2^32).
    const float wres = fmaxf(p - q, 0.f);
    unsigned long long Z;
    unsigned long long f = to_fixed(wres * 2147483648.0f);
    unsigned long long incl = block_incl_scan(f, sWarpU, &Z);
    if (Z == 0) {  // the residual vanished numerically: draw from p_j
      f = to_fixed(p * 2147483648.0f);
      incl = block_incl_scan(f, sWarpU, &Z);
    }
    if (tid == 0) sTok = 0;  // no kept token at all (a row without a finite logit)
    __syncthreads();
    const double u = (double)sU[kb];
    const unsigned long long target = (unsigned long long)(u * (double)Z);  // < Z
    if (f > 0 && incl > target && incl - f <= target) sTok = tok;
    __syncthreads();
    const int drawn = sTok;
    for (int i = tid; i <= k; i += kThreads)
      out[i] = i < j ? a.tokens[(size_t)b * k + i] : (i == j ? drawn : -1);
    if (a.out_probs && tid < k) {  // padded positions are not verified: NaN
      a.out_probs[((size_t)b * k + tid) * 2] = tid < kb ? sP[tid] : NAN;
      a.out_probs[((size_t)b * k + tid) * 2 + 1] = tid < kb ? sQ[tid] : NAN;
    }
    if (tid == 0) {
      a.out_n[b] = j;
      if (a.seq_lens) a.seq_lens[b] += j + 1;
    }
  } else {  // a draft token or the draft length was invalid: fail closed
    for (int i = tid; i <= k; i += kThreads) out[i] = -1;
    if (a.out_probs)
      for (int i = tid; i < 2 * k; i += kThreads) a.out_probs[(size_t)b * 2 * k + i] = NAN;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a.ws.status, SPEC_EBADINDEX);
    }
  }
  // Every call leaves the workspace zero: the kept lists and probabilities.
  __syncthreads();
  for (int i = tid; i < R * K; i += kThreads)
    if (row_used(k, kraw, i / K)) row_words(i / K)[i - (i / K) * K] = 0;
  for (int i = tid; i < 2 * k; i += kThreads) pq[i] = 0.f;
}

__global__ void __launch_bounds__(kThreads) filter_finish_kernel(const ChainArgs a) {
  extern __shared__ unsigned long long sL[];  // nsplit * top_k keys of one row
  const int R = 2 * a.k + 1;
  const int items = a.B * R;
  for (int h = blockIdx.x; h < items; h += gridDim.x) {
    const int b = h / R;
    filter_row_item(a, b, h - b * R, sL);
    __syncthreads();
  }
  // Completion of this grid then implies completion of pass 1.
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// CTAs of the finish grid that fit on the device at once for `smem` bytes
// of dynamic shared memory (the last query is cached).
cudaError_t finish_grid(size_t smem, int* grid) {
  static std::mutex mu;
  static int cdev = -1, cgrid = 0;
  static size_t csmem = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev != cdev || smem != csmem) {
    e = cudaFuncSetAttribute(filter_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, filter_finish_kernel, kThreads,
                                                      smem);
    if (e != cudaSuccess) return e;
    cdev = dev;
    csmem = smem;
    cgrid = sms * (per_sm > 0 ? per_sm : 1);
  }
  *grid = cgrid;
  return cudaSuccess;
}

template <int DT, bool VEC>
cudaError_t launch_filtered_t(const ChainArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(unsigned long long) * (size_t)a.nsplit * a.top_k;
  int slots = 0;
  cudaError_t e = finish_grid(smem, &slots);
  if (e != cudaSuccess) return e;
  const long g1 = (long)a.B * (2 * a.k + 1) * a.nsplit;
  filter_topk_kernel<DT, VEC><<<(unsigned)g1, kThreads, 0, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long items = (long)a.B * (2 * a.k + 1);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(items < slots ? items : slots));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, filter_finish_kernel, a);
}

}  // namespace

cudaError_t launch_filtered(const ChainArgs& a, int dtype, bool vec, cudaStream_t st) {
  if (dtype == SPEC_BF16)
    return vec ? launch_filtered_t<SPEC_BF16, true>(a, st) : launch_filtered_t<SPEC_BF16, false>(a, st);
  return vec ? launch_filtered_t<SPEC_F32, true>(a, st) : launch_filtered_t<SPEC_F32, false>(a, st);
}

}  // namespace sv
