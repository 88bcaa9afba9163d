// Chain rejection-sampling verify (vLLM anatomy page, "Speculative Decoding":
// accept left to right, stop at the first rejection, resample from
// max(0, p - q) normalised, or take a bonus token from the extra row; vLLM
// learning book, section 2: accept iff r < min(1, p(x_i)/q(x_i))).
//
// Pass 1, chain_rowstats_kernel: one short-lived CTA per 32 KB slice of a
// target or draft row.  It reads its slice once with 128-bit loads and
// reduces it to softmax statistics: each warp takes its own max, sums
// 2^(c(x - max)) (c = log2(e)/T) with packed fp32x2 arithmetic and one exp
// per logit, and thread 0 merges the eight warp pairs into the slice's (M, S)
// and publishes it as one 64-bit word (no fence, no counter).  Slices run in
// request order, so requests complete one after another.  No pass-1 CTA
// waits for another.
//
// Pass 2, chain_draw_kernel: launched as a programmatic dependent of pass 1
// (scheduled once every pass-1 CTA has started), one wave of CTAs taking
// draw items (64 or more chunks of 256 tokens of one request, sized so that
// the items of the call fit in one wave where possible) in grid-stride order.
// For each item a CTA gathers x_i's logits, merges its request's slice
// statistics as their words arrive (no grid-wide wait: most requests are
// complete when the grid starts, the rest finish during pass 1's last wave)
// and runs the accept scan (tiny; every CTA of the request repeats it).  It then sums the draw weights of its
// chunks: w_t = max(0, p_j(t) - q_j(t)) after a rejection at j, w_t = p_k(t)
// when all k are accepted, and publishes each chunk sum and the item total in
// 64-bit fixed point.  The request's last item (atomic ticket, no waiting)
// loads every chunk sum at once, finds the chunk holding u*Z with a
// block-wide exact prefix sum, re-reads only that chunk, scans it with a
// warp prefix sum and writes the outputs.
#include <mutex>

#include "kernels.cuh"

namespace sv {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Sum of 2^(c (x - M)) over one vector, as a pair of partial sums.
template <int DT, bool VEC>
__device__ __forceinline__ float2 vec_expsum(const uint32_t (&w)[Io<DT, VEC>::NW], float2 nm,
                                             float2 ch, float2 cl) {
  if constexpr (VEC && DT == SPEC_BF16) {
    float2 e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 d = add2(make_float2(bf16_lo(w[j]), bf16_hi(w[j])), nm);
      const float2 y = fma2(d, ch, mul2(d, cl));
      e[j] = make_float2(ex2(y.x), ex2(y.y));
    }
    return add2(add2(e[0], e[1]), add2(e[2], e[3]));
  } else if constexpr (VEC) {
    float2 e[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float2 d = add2(make_float2(__uint_as_float(w[2 * j]), __uint_as_float(w[2 * j + 1])), nm);
      const float2 y = fma2(d, ch, mul2(d, cl));
      e[j] = make_float2(ex2(y.x), ex2(y.y));
    }
    return add2(e[0], e[1]);
  } else {
    float x[1];
    Io<DT, false>::unpack(w, x);
    return make_float2(ex2(scaled(x[0] + nm.x, ch.x, cl.x)), 0.f);
  }
}

// Slice statistics (M, S) as one 64-bit word: M in the low half, S in the
// high half.  A written word is never 0: a finite M comes with S >= 1 (the
// slice maximum contributes 2^0), M = -inf and NaN have nonzero bits.  So 0
// means "not yet written"; kNoStats stands for an absent slice (-inf, 0).
constexpr unsigned long long kNoStats = 0xff800000ull;
__device__ __forceinline__ unsigned long long stats_pack(float M, float S) {
  return ((unsigned long long)__float_as_uint(S) << 32) | __float_as_uint(M);
}
__device__ __forceinline__ float2 stats_unpack(unsigned long long v) {
  return make_float2(__uint_as_float((uint32_t)v), __uint_as_float((uint32_t)(v >> 32)));
}
__device__ __forceinline__ unsigned long long wait_stats(const ChainArgs& a,
                                                         const unsigned long long* p, bool* to) {
  return wait_word(p, a.ws.status, kNoStats, a.wait_cycles, to);
}

// ------------------------------------------------------------------ pass 1
// Row of slice-row index rr in pass-1 order: request-major, so requests
// finish one after another and most are complete when the draw grid is
// scheduled (during pass 1's last wave).  r < k+1 is target row r, r > k is
// draft row r-k-1.
__device__ __forceinline__ void slice_row(const ChainArgs& a, int rr, int& b, int& r) {
  const int R = 2 * a.k + 1;
  b = rr / R;
  r = rr - b * R;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 6) chain_rowstats_kernel(const ChainArgs a) {
  asm volatile("griddepcontrol.launch_dependents;");
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x;
  const int rr = blockIdx.x / a.nsplit, s = blockIdx.x - rr * a.nsplit;
  int b, r;
  slice_row(a, rr, b, r);
  if (a.draft_lens) {  // ragged: rows past the request's draft length are not verified
    const int kb = a.draft_lens[b];
    if (kb < 0 || kb > a.k || (r <= a.k ? r > kb : r - a.k - 1 >= kb)) return;
  }
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
  const int vbeg = s * a.vps;
  const int vend = min(a.nvec, vbeg + a.vps);

  uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + tid + u * kThreads;
    if (v < vend) IO::load(row, v, w[u]);
  }
  float m = -INFINITY;
  if constexpr (VEC && DT == SPEC_BF16) {
    uint32_t mx = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u)
      if (vbeg + tid + u * kThreads < vend)
        mx = bf16x2_max(mx, bf16x2_max(bf16x2_max(w[u][0], w[u][1]), bf16x2_max(w[u][2], w[u][3])));
    m = fmaxf(bf16_lo(mx), bf16_hi(mx));
  } else {
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u)
      if (vbeg + tid + u * kThreads < vend) m = fmaxf(m, IO::vmax(w[u]));
  }
  // Warp max, then this warp's sum relative to it; thread 0 merges the warps.
  __shared__ float s_wm[kWarps], s_ws[kWarps];
  const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float Ms = m == -INFINITY ? 0.f : m;
  const float2 nm = make_float2(-Ms, -Ms), ch = make_float2(a.c_hi, a.c_hi),
               cl = make_float2(a.c_lo, a.c_lo);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u)
    if (vbeg + tid + u * kThreads < vend) acc = add2(acc, vec_expsum<DT, VEC>(w[u], nm, ch, cl));
  const float ssum = warp_sum(acc.x + acc.y);
  if (lane == 0) {
    s_wm[warp] = m;
    s_ws[warp] = ssum;
  }
  __syncthreads();
  if (tid == 0) {
    float M = s_wm[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) M = fmaxf(M, s_wm[i]);
    float S = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kWarps; ++i)
        if (s_ws[i] > 0.f) S += s_ws[i] * ex2(scaled(s_wm[i] - M, a.c_hi, a.c_lo));
    }
    // One 64-bit store publishes the pair; the draw polls for it (no fence).
    st_relaxed_u64(a.ws.stats + ((size_t)b * (2 * a.k + 1) + r) * a.nsplit + s, stats_pack(M, S));
  }
}

// ------------------------------------------------------------------ pass 2
// The 8 draw weights of lane `lane` in chunk `c` (0 past the row's end):
// residual: 2^(c(xp - mp)) - lam * 2^(c(xq - mq)) clamped at 0, lam = Sp/Sq
// (that is Sp * max(0, p - q)); bonus (qrow == nullptr): 2^(c(xp - mp)).
template <int DT, bool VEC>
__device__ __forceinline__ void chunk_weights(const char* prow, const char* qrow, int c, int lane,
                                              int V, float mp, float mq, float lam, float c_hi,
                                              float c_lo, float (&wv)[8]) {
  const long t0 = (long)c * kChunk + lane * 8;
  float xp[8], xq[8];
  if constexpr (VEC) {
    constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
    constexpr int LOADS = 8 * ES / 16;  // 16-byte loads per row per lane
    using IO = Io<DT, true>;
    uint32_t P[LOADS][4], Q[LOADS][4];
#pragma unroll
    for (int h = 0; h < LOADS; ++h) {  // issue every load first
      const long th = t0 + h * IO::EPV;
      if (th < V) {
        ld_stream_v4(prow + th * ES, P[h]);
        if (qrow) ld_stream_v4(qrow + th * ES, Q[h]);
      }
    }
#pragma unroll
    for (int h = 0; h < LOADS; ++h) {
      const long th = t0 + h * IO::EPV;
      float ep[IO::EPV], eq[IO::EPV];
      if (th < V) {
        IO::unpack(P[h], ep);
        if (qrow) IO::unpack(Q[h], eq);
      } else {
#pragma unroll
        for (int i = 0; i < IO::EPV; ++i) ep[i] = eq[i] = -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < IO::EPV; ++i) {
        xp[h * IO::EPV + i] = ep[i];
        xq[h * IO::EPV + i] = qrow ? eq[i] : -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const long t = t0 + i;
      xp[i] = t < V ? load_logit<DT>(prow, t) : -INFINITY;
      xq[i] = (qrow && t < V) ? load_logit<DT>(qrow, t) : -INFINITY;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float ep = ex2(scaled(xp[i] - mp, c_hi, c_lo));
    if (qrow) {
      const float eq = ex2(scaled(xq[i] - mq, c_hi, c_lo));
      wv[i] = fmaxf(fmaf(-lam, eq, ep), 0.f);
    } else {
      wv[i] = ep;
    }
  }
}

// Warp-wide inclusive prefix sum of 64-bit values.
__device__ __forceinline__ unsigned long long warp_incl_u64(unsigned long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

__device__ __forceinline__ float tree8(const float (&v)[8]) {
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// Draw weights of one 16-byte vector pair of bf16 (8 tokens) with packed
// fp32x2 arithmetic; the same operations as chunk_weights, lane by lane.
__device__ __forceinline__ void weights8_bf16(const uint32_t (&P)[4], const uint32_t (&Q)[4],
                                              bool resid, float2 nmp, float2 nmq, float2 nlam,
                                              float2 ch, float2 cl, float (&wv)[8]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 dp = add2(make_float2(bf16_lo(P[j]), bf16_hi(P[j])), nmp);
    const float2 yp = fma2(dp, ch, mul2(dp, cl));
    const float2 ep = make_float2(ex2(yp.x), ex2(yp.y));
    if (resid) {
      const float2 dq = add2(make_float2(bf16_lo(Q[j]), bf16_hi(Q[j])), nmq);
      const float2 yq = fma2(dq, ch, mul2(dq, cl));
      const float2 eq = make_float2(ex2(yq.x), ex2(yq.y));
      const float2 w = fma2(nlam, eq, ep);
      wv[2 * j] = fmaxf(w.x, 0.f);
      wv[2 * j + 1] = fmaxf(w.y, 0.f);
    } else {
      wv[2 * j] = ep.x;
      wv[2 * j + 1] = ep.y;
    }
  }
}

// Draw-weight sums of chunks [c0, c1) (warp w takes c0+w, c0+w+8, ...).
// Each warp issues the loads of four chunks before using any.  The weights
// are those of chunk_weights, computed with the same operations.
// Returns, in lane 0 of each warp, the fixed-point total of that warp's chunks.
template <int DT, bool VEC>
__device__ __forceinline__ unsigned long long chunk_sums(const ChainArgs& a, const char* prow,
                                                         const char* qrow, int c0, int c1, float mp,
                                                         float mq, float lam,
                                                         unsigned long long* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long wtot = 0;
  if constexpr (VEC && DT == SPEC_BF16) {
    constexpr int GRP = 4;
    const bool resid = qrow != nullptr;
    const float2 nmp = make_float2(-mp, -mp), nmq = make_float2(-mq, -mq),
                 nlam = make_float2(-lam, -lam), ch = make_float2(a.c_hi, a.c_hi),
                 cl = make_float2(a.c_lo, a.c_lo);
#pragma unroll 1
    for (int cb = c0 + warp; cb < c1; cb += GRP * kWarps) {
      uint32_t P[GRP][4], Q[GRP][4];
#pragma unroll
      for (int i = 0; i < GRP; ++i) {
        const int c = cb + i * kWarps;
        const long t = (long)c * kChunk + lane * 8;
        if (c < c1 && t < a.V) {
          ld_stream_v4(prow + t * 2, P[i]);
          if (resid) ld_stream_v4(qrow + t * 2, Q[i]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) P[i][e] = Q[i][e] = 0xff80ff80u;  // -inf: zero weight
        }
      }
#pragma unroll
      for (int i = 0; i < GRP; ++i) {
        const int c = cb + i * kWarps;
        if (c >= c1) continue;
        float wv[8];
        weights8_bf16(P[i], Q[i], resid, nmp, nmq, nlam, ch, cl, wv);
        const unsigned long long f = to_fixed(warp_sum(tree8(wv)));
        if (lane == 0) out[c] = f;
        wtot += f;
      }
    }
  } else {
    for (int c = c0 + warp; c < c1; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC>(prow, qrow, c, lane, a.V, mp, mq, lam, a.c_hi, a.c_lo, wv);
      const unsigned long long f = to_fixed(warp_sum(tree8(wv)));
      if (lane == 0) out[c] = f;
      wtot += f;
    }
  }
  return wtot;
}

// The request's last CTA: locate u*Z among the chunk sums (one round trip for
// all of them), re-read and scan that chunk, return the token (all threads
// call it; the result is valid in every thread).
template <int DT, bool VEC>
__device__ int draw_token(const ChainArgs& a, int b, const char* prow, const char* qrow,
                          float mp, float mq, float lam, double u) {
  __shared__ unsigned long long sTarget, sPre, sZ;
  __shared__ unsigned long long sWarpTot[kWarps];
  __shared__ int sChunk, sTok, sRetry, sLastPos;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.nchunks, ni = a.nsplit2;
  unsigned long long* chunks = a.ws.chunks + (size_t)b * n;
  unsigned long long* items = a.ws.items + (size_t)b * ni;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // One round trip: every thread loads two chunk sums while warp 0 adds
    // the item totals into the exact total Z.
    unsigned long long v0 = 2 * tid < n ? __ldcg(chunks + 2 * tid) : 0;
    unsigned long long v1 = 2 * tid + 1 < n ? __ldcg(chunks + 2 * tid + 1) : 0;
    if (warp == 0) {
      unsigned long long t = 0;
      for (int i = lane; i < ni; i += 32) t += __ldcg(items + i);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
      if (lane == 0) {
        sZ = t;
        sRetry = t == 0;
        sTarget = t ? (unsigned long long)(u * (double)t) : 0;  // < Z: u < 1
        sChunk = -1;
        sLastPos = -1;
      }
    }
    __syncthreads();
    if (!sRetry) {
      // The chunk holding the target: block-wide exact prefix sums, 2 * kThreads
      // chunks at a time; exactly one thread sees the running sum cross it.
      const unsigned long long target = sTarget;
      unsigned long long carry = 0;
      for (int base = 0; base < n; base += 2 * kThreads) {
        const int i0 = base + 2 * tid;
        if (base > 0) {
          v0 = i0 < n ? __ldcg(chunks + i0) : 0;
          v1 = i0 + 1 < n ? __ldcg(chunks + i0 + 1) : 0;
        }
        const unsigned long long mine = v0 + v1;
        const unsigned long long incl = warp_incl_u64(mine);
        if (lane == 31) sWarpTot[warp] = incl;
        __syncthreads();
        unsigned long long wbase = 0, seg = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const unsigned long long t = sWarpTot[w];
          wbase += w < warp ? t : 0;
          seg += t;
        }
        const unsigned long long lb = carry + wbase + incl - mine;  // before chunk i0
        if (v0 > 0 && lb <= target && lb + v0 > target) {
          sChunk = i0;
          sPre = lb;
        } else if (v1 > 0 && lb + v0 <= target && lb + mine > target) {
          sChunk = i0 + 1;
          sPre = lb + v0;
        }
        if (mine > 0) atomicMax(&sLastPos, v1 > 0 ? i0 + 1 : i0);
        __syncthreads();
        if (sChunk >= 0) break;
        carry += seg;
        __syncthreads();  // sWarpTot is rewritten next
      }
      if (sChunk < 0 && tid == 0) {  // not reached while u < 1: the last positive chunk
        const int c = sLastPos < 0 ? 0 : sLastPos;
        sChunk = c;
        sPre = sZ - __ldcg(chunks + c);
      }
      __syncthreads();
      break;
    }
    // The residual vanished numerically: draw from p_j instead (this CTA
    // recomputes every chunk and item sum; a rare path).
    qrow = nullptr;
    lam = 0.f;
    for (int c = warp; c < n; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC>(prow, nullptr, c, lane, a.V, mp, 0.f, 0.f, a.c_hi, a.c_lo, wv);
      const unsigned long long f = to_fixed(warp_sum(tree8(wv)));
      if (lane == 0) chunks[c] = f;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      for (int i = 0; i < ni; ++i) {
        unsigned long long t = 0;
        for (int c = i * a.cpc; c < min(n, (i + 1) * a.cpc); ++c) t += __ldcg(chunks + c);
        items[i] = t;
      }
      __threadfence();
    }
    __syncthreads();
  }
  if (tid == 0 && sChunk < 0) {  // Z stayed 0 after the retry (not reached): chunk 0
    sChunk = 0;
    sPre = 0;
  }
  __syncthreads();
  if (warp == 0) {
    const int c = sChunk;
    float wv[8];
    chunk_weights<DT, VEC>(prow, qrow, c, lane, a.V, mp, mq, lam, a.c_hi, a.c_lo, wv);
    float loc[8];
    loc[0] = wv[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) loc[i] = loc[i - 1] + wv[i];
    float incl = loc[7];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const unsigned long long pre = sPre, target = sTarget;
    int first = 8;
#pragma unroll
    for (int i = 7; i >= 0; --i)
      if (wv[i] > 0.f && pre + to_fixed(excl + loc[i]) > target) first = i;
    const unsigned hit = __ballot_sync(0xffffffffu, first < 8);
    int tok;
    if (hit) {
      const int L = __ffs(hit) - 1;
      tok = c * kChunk + L * 8 + __shfl_sync(0xffffffffu, first, L);
    } else {  // rounding left u*Z past this chunk's scan: last positive weight
      int last = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (wv[i] > 0.f) last = i;
      const unsigned any = __ballot_sync(0xffffffffu, last >= 0);
      const int L = any ? 31 - __clz(any) : 0;
      const int e = __shfl_sync(0xffffffffu, last, L);
      tok = c * kChunk + L * 8 + (e < 0 ? 0 : e);
    }
    if (lane == 0) sTok = tok;
  }
  __syncthreads();
  // Every call leaves the workspace zero: clear this request's sums.
  for (int i = tid; i < n; i += kThreads) chunks[i] = 0;
  for (int i = tid; i < ni; i += kThreads) items[i] = 0;
  return sTok;
}

template <int DT, bool VEC>
__device__ __forceinline__ void draw_item(const ChainArgs& a, int b, int part) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  __shared__ float sM[2 * SPEC_MAX_DRAFT + 1], sS[2 * SPEC_MAX_DRAFT + 1];
  __shared__ float sP[SPEC_MAX_DRAFT], sQ[SPEC_MAX_DRAFT], sU[SPEC_MAX_DRAFT + 1];
  __shared__ int sJ, sBad, sLast, sFailed;
  __shared__ unsigned long long sWT[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k, R = 2 * k + 1;
  const size_t row_bytes = (size_t)a.V * ES;

  // Ragged verify: this request has kb <= k real drafts; rows past them were
  // not streamed and are not read.  A length outside [0, k] fails closed.
  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const bool bad_len = kraw < 0 || kraw > k;
  const int kb = bad_len ? 0 : kraw;
  // Gather the logits of x_i (inputs only, so before the wait on pass 1).
  float xp = 0.f, xq = 0.f;
  bool bad = bad_len;
  if (tid < kb) {
    const int x = a.tokens[(size_t)b * k + tid];
    bad = x < 0 || x >= a.V;
    if (!bad) {
      xp = load_logit<DT>(a.target + ((size_t)b * (k + 1) + tid) * row_bytes, x);
      xq = load_logit<DT>(a.draft + ((size_t)b * k + tid) * row_bytes, x);
    }
  }
  if (tid <= k)
    sU[tid] = a.uniforms ? a.uniforms[(size_t)b * (k + 1) + tid]
                         : philox_uniform(a.seeds[b], a.offsets[b], tid);
  if (tid == 0) sBad = bad_len;
  // Rows this request verifies: target rows 0..kb, draft rows 0..kb-1.
  auto used = [&](int r) { return r <= k ? r <= kb : r - k - 1 < kb; };
  const int rows = bad_len ? 0 : R;
  // Merge the slice statistics of every row of the request, in a fixed
  // order, as they arrive: warp w takes rows w, w+8, ...; it issues the loads
  // of four rows' words before using any (waiting only for words still 0),
  // takes each row max with shuffles, then adds S_s * 2^(c(m_s - M)) with one
  // exp per slice (no chain of exps).
  const unsigned long long* sb = a.ws.stats + (size_t)b * R * a.nsplit;
  bool to = false;  // a wait of this thread ran out
  for (int r0 = warp; r0 < rows; r0 += 4 * kWarps) {
    unsigned long long v[4][2];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int u = lane + 32 * h;
        v[q][h] = (r < R && used(r) && u < a.nsplit) ? ld_relaxed_u64(sb + (size_t)r * a.nsplit + u)
                                                     : kNoStats;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (!v[q][h])  // only a present slice reads 0
          v[q][h] = wait_stats(a, sb + (size_t)(r0 + q * kWarps) * a.nsplit + lane + 32 * h, &to);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = r0 + q * kWarps;
      if (r >= R || !used(r)) continue;  // the same for the whole warp
      const unsigned long long* pr = sb + (size_t)r * a.nsplit;
      const float2 e0 = stats_unpack(v[q][0]), e1 = stats_unpack(v[q][1]);
      float m = fmaxf(e0.x, e1.x);
      for (int u = lane + 64; u < a.nsplit; u += 32)
        m = fmaxf(m, stats_unpack(wait_stats(a, pr + u, &to)).x);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float sum = 0.f;
      if (m != -INFINITY) {
        if (e0.y > 0.f) sum += e0.y * ex2(scaled(e0.x - m, a.c_hi, a.c_lo));
        if (e1.y > 0.f) sum += e1.y * ex2(scaled(e1.x - m, a.c_hi, a.c_lo));
        for (int u = lane + 64; u < a.nsplit; u += 32) {
          const float2 e = stats_unpack(ld_relaxed_u64(pr + u));  // written: seen above
          if (e.y > 0.f) sum += e.y * ex2(scaled(e.x - m, a.c_hi, a.c_lo));
        }
      }
      sum = warp_sum(sum);
      if (lane == 0) {
        sM[r] = m;
        sS[r] = sum;
      }
    }
  }
  // A statistics word that never arrived: this item skips its draw work and
  // the request fails closed (every item's flag reaches the finishing item
  // through the ticket below).
  if (__syncthreads_or(to) && tid == 0) {
    sBad = 1;
    atomicExch(&a.ws.sync[b].failed, 1);
  }
  if (tid < kb) {
    if (bad) {
      sBad = 1;
    } else {
      sP[tid] = ex2(scaled(xp - sM[tid], a.c_hi, a.c_lo)) / sS[tid];
      sQ[tid] = ex2(scaled(xq - sM[k + 1 + tid], a.c_hi, a.c_lo)) / sS[k + 1 + tid];
    }
  }
  __syncthreads();
  if (warp == 0) {  // accept scan: r_i < p_i(x_i) / q_i(x_i), q == 0 accepts; j = first reject
    unsigned rej[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = lane + 32 * h;
      bool rj = false;
      if (i < kb) {
        const float ratio = sQ[i] > 0.f ? sP[i] / sQ[i] : INFINITY;
        rj = !(sU[i] < ratio);
      }
      rej[h] = __ballot_sync(0xffffffffu, rj);
    }
    if (lane == 0)
      sJ = sBad ? -1 : rej[0] ? __ffs(rej[0]) - 1 : rej[1] ? 31 + __ffs(rej[1]) : kb;
  }
  __syncthreads();
  const int j = sJ;
  const char* prow = nullptr;
  const char* qrow = nullptr;
  float mp = 0.f, mq = 0.f, lam = 0.f;
  if (j >= 0) {
    prow = a.target + ((size_t)b * (k + 1) + j) * row_bytes;
    mp = sM[j];
    if (j < kb) {
      qrow = a.draft + ((size_t)b * k + j) * row_bytes;
      mq = sM[k + 1 + j];
      lam = sS[j] / sS[k + 1 + j];
    }
    const int c0 = part * a.cpc, c1 = min(a.nchunks, c0 + a.cpc);
    const unsigned long long wt =
        chunk_sums<DT, VEC>(a, prow, qrow, c0, c1, mp, mq, lam, a.ws.chunks + (size_t)b * a.nchunks);
    if (lane == 0) sWT[warp] = wt;
    __syncthreads();
    if (tid == 0) {  // the item's total (exact in fixed point) for the two-level search
      unsigned long long t = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) t += sWT[w];
      a.ws.items[(size_t)b * a.nsplit2 + part] = t;
    }
  }
  if (lane == 0) __threadfence();
  __syncthreads();
  if (tid == 0) {
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
  // Every item has merged: return the request's statistics words to 0.
  for (int i = tid; i < R * a.nsplit; i += kThreads)
    const_cast<unsigned long long*>(sb)[i] = 0;
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (j < 0 || sFailed) {  // a bad draft token or length, or a wait ran out: fail closed
    for (int i = tid; i < a.nchunks; i += kThreads) a.ws.chunks[(size_t)b * a.nchunks + i] = 0;
    for (int i = tid; i < a.nsplit2; i += kThreads) a.ws.items[(size_t)b * a.nsplit2 + i] = 0;
    for (int i = tid; i <= k; i += kThreads) out[i] = -1;
    if (a.out_probs)
      for (int i = tid; i < 2 * k; i += kThreads) a.out_probs[(size_t)b * 2 * k + i] = NAN;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a.ws.status, SPEC_EBADINDEX);
    }
    return;
  }
  if (a.out_probs && tid < k) {  // padded positions are not verified: NaN
    a.out_probs[((size_t)b * k + tid) * 2] = tid < kb ? sP[tid] : NAN;
    a.out_probs[((size_t)b * k + tid) * 2 + 1] = tid < kb ? sQ[tid] : NAN;
  }
  const double u = (double)sU[kb];
  const int tok = draw_token<DT, VEC>(a, b, prow, qrow, mp, mq, lam, u);
  for (int i = tid; i <= k; i += kThreads)
    out[i] = i < j ? a.tokens[(size_t)b * k + i] : (i == j ? tok : -1);
  if (tid == 0) {
    a.out_n[b] = j;
    if (a.seq_lens) a.seq_lens[b] += j + 1;
  }
}



template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) chain_draw_kernel(const ChainArgs a) {
  const int items = a.B * a.nsplit2;
  for (int h = blockIdx.x; h < items; h += gridDim.x) {
    const int b = h / a.nsplit2;
    draw_item<DT, VEC>(a, b, h - b * a.nsplit2);
    __syncthreads();  // shared state of this item is no longer read
  }
  // Completion of this grid then implies completion of pass 1, which stream
  // order relies on (nothing above waits for the whole of pass 1).
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

template <int DT, bool VEC>
cudaError_t draw_grid(int* grid) {
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_draw_kernel<DT, VEC>, kThreads, 0);
    if (e != cudaSuccess) return e;
    cached[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  *grid = cached[dev];
  return cudaSuccess;
}

template <int DT, bool VEC>
cudaError_t launch_chain_t(const ChainArgs& args, cudaStream_t st, bool skip_pass1) {
  int slots = 0;
  cudaError_t e = draw_grid<DT, VEC>(&slots);
  if (e != cudaSuccess) return e;
  // Draw item size: 64 chunks, doubled until every item fits in one wave of
  // draw CTAs.  Each item pays the merge and accept-scan latency once, so
  // with many requests fewer, larger items finish sooner; with few, smaller
  // items spread each request over more SMs.
  ChainArgs a = args;
  while ((long)a.B * a.nsplit2 > slots && a.cpc < a.nchunks) {
    a.cpc *= 2;
    a.nsplit2 = ceil_div(a.nchunks, a.cpc);
  }
  const long g1 = (long)a.B * (2 * a.k + 1) * a.nsplit;
  if (!skip_pass1) {
    chain_rowstats_kernel<DT, VEC><<<(unsigned)g1, kThreads, 0, st>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long items = (long)a.B * a.nsplit2;
  // Pass 2 may be scheduled once every pass-1 CTA has started; each draw
  // item waits only for its own request's slices.
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
  return cudaLaunchKernelEx(&cfg, chain_draw_kernel<DT, VEC>, a);
}

}  // namespace

cudaError_t launch_chain(const ChainArgs& a, int dtype, bool vec, cudaStream_t st, bool skip_pass1) {
  if (dtype == SPEC_BF16)
    return vec ? launch_chain_t<SPEC_BF16, true>(a, st, skip_pass1)
               : launch_chain_t<SPEC_BF16, false>(a, st, skip_pass1);
  return vec ? launch_chain_t<SPEC_F32, true>(a, st, skip_pass1)
             : launch_chain_t<SPEC_F32, false>(a, st, skip_pass1);
}

}  // namespace sv
