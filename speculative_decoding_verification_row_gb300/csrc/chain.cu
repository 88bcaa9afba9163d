// Chain rejection-sampling verify (vLLM anatomy page, "Speculative Decoding":
// accept left to right, stop at the first rejection, resample from
// max(0, p - q) normalised, or take a bonus token from the extra row; vLLM
// learning book, section 2: accept iff r < min(1, p(x_i)/q(x_i))).
//
// Pass 1, chain_stats_kernel: one CTA per (request, row, unit) streams its
// slice of a target or draft row once and reduces it to the softmax statistics
// (max m, S = sum 2^(log2(e)/T * (x - m))).  The request's last CTA merges the
// units of all 2k+1 rows, gathers p_i(x_i) and q_i(x_i), and runs the
// accept scan; it stores the stopping position and the statistics of the
// row(s) the final draw needs.
//
// Pass 2, chain_sample_kernel: the final token is drawn by inverse CDF from
// w_t = max(0, p_j(t) - q_j(t)) (rejection at j) or w_t = p_k(t) (bonus).
// CTAs of a request split the row(s) into 256-token chunks and store each
// chunk's weight sum; the request's last CTA prefix-sums the chunk sums in
// fp64, finds the chunk holding u * Z, re-reads only that chunk and scans it
// with a warp prefix sum to find the token.
#include "kernels.cuh"

namespace sv {

// Block-wide merge of (m, s); the result is valid in thread 0.
__device__ __forceinline__ void block_lse(float& m, float& s, float c_hi, float c_lo) {
  __shared__ float sm[kWarps], ss[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off),
              c_hi, c_lo);
  if (lane == 0) {
    sm[warp] = m;
    ss[warp] = s;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kWarps ? sm[lane] : -INFINITY;
    s = lane < kWarps ? ss[lane] : 0.f;
#pragma unroll
    for (int off = kWarps / 2; off > 0; off >>= 1)
      lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off),
                c_hi, c_lo);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ------------------------------------------------------------------ pass 1 epilogue
template <int DT>
__device__ void chain_scan(const ChainArgs& a, int b) {
  __shared__ float sM[2 * SPEC_MAX_DRAFT + 1], sS[2 * SPEC_MAX_DRAFT + 1];
  __shared__ float sRatio[SPEC_MAX_DRAFT];
  __shared__ int sBad;
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const int k = a.k, R = 2 * k + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) sBad = 0;
  // Merge the units of every row, in unit order.
  for (int r = warp; r < R; r += kWarps) {
    float m = -INFINITY, s = 0.f;
    const float2* pr = a.ws.part + ((size_t)b * R + r) * a.nsplit;
    for (int u = lane; u < a.nsplit; u += 32) {
      const float2 v = __ldcg(pr + u);
      lse_merge(m, s, v.x, v.y, a.c_hi, a.c_lo);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, off), __shfl_xor_sync(0xffffffffu, s, off),
                a.c_hi, a.c_lo);
    if (lane == 0) {
      sM[r] = m;
      sS[r] = s;
    }
  }
  __syncthreads();
  const size_t row_bytes = (size_t)a.V * ES;
  for (int i = threadIdx.x; i < k; i += kThreads) {
    const int x = a.tokens[(size_t)b * k + i];
    if (x < 0 || x >= a.V) {
      sBad = 1;
      sRatio[i] = 0.f;
      continue;
    }
    const float xp = load_logit<DT>(a.target + ((size_t)b * (k + 1) + i) * row_bytes, x);
    const float xq = load_logit<DT>(a.draft + ((size_t)b * k + i) * row_bytes, x);
    const float p = ex2(scaled(xp - sM[i], a.c_hi, a.c_lo)) / sS[i];
    const float q = ex2(scaled(xq - sM[k + 1 + i], a.c_hi, a.c_lo)) / sS[k + 1 + i];
    if (a.out_probs) {
      a.out_probs[((size_t)b * k + i) * 2] = p;
      a.out_probs[((size_t)b * k + i) * 2 + 1] = q;
    }
    sRatio[i] = q > 0.f ? p / q : INFINITY;
  }
  __syncthreads();
  if (sBad) {
    if (a.out_probs)
      for (int i = threadIdx.x; i < 2 * k; i += kThreads) a.out_probs[(size_t)b * 2 * k + i] = NAN;
    if (threadIdx.x == 0) {
      set_status(a.ws.status, SPEC_EBADINDEX);
      ReqInfo ri{};
      ri.j = -1;
      a.ws.req[b] = ri;
    }
    return;
  }
  if (threadIdx.x == 0) {
    const float* r = a.uniforms + (size_t)b * (k + 1);
    int j = k;
    for (int i = 0; i < k; ++i)
      if (!(r[i] < sRatio[i])) {
        j = i;
        break;
      }
    ReqInfo ri{};
    ri.j = j;
    ri.mp = sM[j];
    ri.sp = sS[j];
    if (j < k) {
      ri.mq = sM[k + 1 + j];
      ri.sq = sS[k + 1 + j];
    }
    a.ws.req[b] = ri;
  }
}

// ------------------------------------------------------------------ pass 1
template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) chain_stats_kernel(const ChainArgs a) {
  using IO = Io<DT, VEC>;
  const int R = 2 * a.k + 1;
  const int per_req = R * a.nsplit;
  const int b = blockIdx.x / per_req;
  const int rem = blockIdx.x - b * per_req;
  const int r = rem / a.nsplit;
  const int s = rem - r * a.nsplit;
  const size_t row_bytes = (size_t)a.V * IO::ES;
  const char* row = r <= a.k ? a.target + ((size_t)b * (a.k + 1) + r) * row_bytes
                             : a.draft + ((size_t)b * a.k + (r - a.k - 1)) * row_bytes;
  const int vbeg = s * a.vps;
  const int vend = min(a.nvec, vbeg + a.vps);

  uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + (int)threadIdx.x + u * kThreads;
    if (v < vend) IO::load(row, v, w[u]);
  }
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + (int)threadIdx.x + u * kThreads;
    if (v < vend) m = fmaxf(m, IO::vmax(w[u]));
  }
  const float ms = m == -INFINITY ? 0.f : m;
  float acc = 0.f;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + (int)threadIdx.x + u * kThreads;
    if (v < vend) {
      float e[IO::EPV];
      IO::unpack(w[u], e);
#pragma unroll
      for (int i = 0; i < IO::EPV; ++i) e[i] = ex2(scaled(e[i] - ms, a.c_hi, a.c_lo));
#pragma unroll
      for (int h = IO::EPV / 2; h > 0; h >>= 1)
#pragma unroll
        for (int i = 0; i < h; ++i) e[i] += e[i + h];
      acc += e[0];
    }
  }
  block_lse(m, acc, a.c_hi, a.c_lo);
  if (threadIdx.x == 0) a.ws.part[blockIdx.x] = make_float2(m, acc);
  if (!last_arrival(a.ws.tick1 + b, per_req)) return;
  chain_scan<DT>(a, b);
}

// ------------------------------------------------------------------ pass 2
// The 8 draw weights of lane `lane` in chunk `c` (0 past the row's end):
// residual: 2^(c(xp - mp)) - lam * 2^(c(xq - mq)) clamped at 0, lam = Sp/Sq
// (that is Sp * max(0, p - q)); bonus: 2^(c(xp - mp)) (Sp * p).
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
#pragma unroll
    for (int h = 0; h < LOADS; ++h) {
      const long th = t0 + h * IO::EPV;
      float ep[IO::EPV], eq[IO::EPV];
      if (th < V) {
        uint32_t w[4];
        ld_stream_v4(prow + th * ES, w);
        IO::unpack(w, ep);
        if (qrow) {
          ld_stream_v4(qrow + th * ES, w);
          IO::unpack(w, eq);
        }
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

__device__ __forceinline__ float tree8(const float (&v)[8]) {
  return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// Epilogue of pass 2: find the token and write the request's outputs.
template <int DT, bool VEC>
__device__ void chain_finish(const ChainArgs& a, int b, const ReqInfo& ri, const char* prow,
                             const char* qrow, float lam) {
  __shared__ double sTarget, sPre;
  __shared__ int sChunk, sTok, sRetry;
  const int k = a.k, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j = ri.j;
  float* chunks = a.ws.chunks + (size_t)b * a.nchunks;
  if (j < 0) {  // failed request: nothing is emitted and the cursor does not move
    for (int i = threadIdx.x; i <= k; i += kThreads) a.out_tokens[(size_t)b * (k + 1) + i] = -1;
    if (threadIdx.x == 0) a.out_n[b] = -1;
    return;
  }
  const double u = (double)a.uniforms[(size_t)b * (k + 1) + k];
  if (threadIdx.x == 0) {
    sChunk = 0;
    sPre = 0.0;
    sTarget = 0.0;
    sRetry = 0;
  }
  __syncthreads();
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (warp == 0) {
      // fp64 prefix over chunk sums: lane l owns a contiguous run of chunks.
      const int n = a.nchunks, per = (n + 31) / 32;
      const int c_lo = min(n, lane * per), c_hi = min(n, c_lo + per);
      double tot = 0.0;
      for (int c = c_lo; c < c_hi; ++c) tot += (double)__ldcg(chunks + c);
      double incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const double Z = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) sRetry = !(Z > 0.0);
      if (Z > 0.0) {
        const double target = u * Z;
        const unsigned hit = __ballot_sync(0xffffffffu, incl > target);
        const unsigned pos = __ballot_sync(0xffffffffu, tot > 0.0);
        const int L = hit ? __ffs(hit) - 1 : 31 - __clz(pos);  // u*Z >= Z only if u >= 1
        if (lane == L) {
          double pre = incl - tot;
          int chosen = -1;
          double chosen_pre = pre;
          for (int c = c_lo; c < c_hi; ++c) {
            const double v = (double)__ldcg(chunks + c);
            if (v > 0.0) {
              chosen = c;  // keeps the last positive chunk if rounding finds none
              chosen_pre = pre;
            }
            if (pre + v > target && v > 0.0) break;
            pre += v;
          }
          sChunk = chosen;
          sPre = chosen_pre;
          sTarget = target;
        }
      }
    }
    __syncthreads();
    if (!sRetry) break;
    // The residual vanished numerically: draw from p_j instead (every CTA
    // chunk sum is recomputed here by this CTA; a rare path).
    qrow = nullptr;
    lam = 0.f;
    for (int c = warp; c < a.nchunks; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC>(prow, nullptr, c, lane, a.V, ri.mp, 0.f, 0.f, a.c_hi, a.c_lo, wv);
      const float s = warp_sum(tree8(wv));
      if (lane == 0) chunks[c] = s;
    }
    __threadfence();
    __syncthreads();
  }
  if (warp == 0) {
    const int c = sChunk;
    float wv[8];
    chunk_weights<DT, VEC>(prow, qrow, c, lane, a.V, ri.mp, ri.mq, lam, a.c_hi, a.c_lo, wv);
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
    const double pre = sPre, target = sTarget;
    int first = 8;
#pragma unroll
    for (int i = 7; i >= 0; --i)
      if (wv[i] > 0.f && pre + (double)(excl + loc[i]) > target) first = i;
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
  const int tok = sTok;
  for (int i = threadIdx.x; i <= k; i += kThreads)
    a.out_tokens[(size_t)b * (k + 1) + i] =
        i < j ? a.tokens[(size_t)b * k + i] : (i == j ? tok : -1);
  if (threadIdx.x == 0) {
    a.out_n[b] = j;
    if (a.seq_lens) a.seq_lens[b] += j + 1;
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) chain_sample_kernel(const ChainArgs a) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const int b = blockIdx.x / a.nsplit2;
  const int sp = blockIdx.x - b * a.nsplit2;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  ReqInfo ri;
  {
    const int4 w0 = __ldcg(reinterpret_cast<const int4*>(a.ws.req + b));
    const int4 w1 = __ldcg(reinterpret_cast<const int4*>(a.ws.req + b) + 1);
    ri.j = w0.x;
    ri.mp = __int_as_float(w0.z);
    ri.sp = __int_as_float(w0.w);
    ri.mq = __int_as_float(w1.x);
    ri.sq = __int_as_float(w1.y);
  }
  const size_t row_bytes = (size_t)a.V * ES;
  const int j = ri.j;
  const char* prow = nullptr;
  const char* qrow = nullptr;
  float lam = 0.f;
  if (j >= 0) {
    prow = a.target + ((size_t)b * (a.k + 1) + j) * row_bytes;
    if (j < a.k) {
      qrow = a.draft + ((size_t)b * a.k + j) * row_bytes;
      lam = ri.sp / ri.sq;
    }
    const int c0 = sp * a.cpc, c1 = min(a.nchunks, c0 + a.cpc);
    for (int c = c0 + warp; c < c1; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC>(prow, qrow, c, lane, a.V, ri.mp, ri.mq, lam, a.c_hi, a.c_lo, wv);
      const float s = warp_sum(tree8(wv));
      if (lane == 0) a.ws.chunks[(size_t)b * a.nchunks + c] = s;
    }
  }
  if (!last_arrival(a.ws.tick2 + b, a.nsplit2)) return;
  chain_finish<DT, VEC>(a, b, ri, prow, qrow, lam);
}

// ------------------------------------------------------------------ launch
template <int DT, bool VEC>
cudaError_t launch_chain_t(const ChainArgs& a, cudaStream_t st) {
  const long g1 = (long)a.B * (2 * a.k + 1) * a.nsplit;
  chain_stats_kernel<DT, VEC><<<(unsigned)g1, kThreads, 0, st>>>(a);
  const long g2 = (long)a.B * a.nsplit2;
  chain_sample_kernel<DT, VEC><<<(unsigned)g2, kThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_chain(const ChainArgs& a, int dtype, bool vec, cudaStream_t st) {
  if (dtype == SPEC_BF16)
    return vec ? launch_chain_t<SPEC_BF16, true>(a, st) : launch_chain_t<SPEC_BF16, false>(a, st);
  return vec ? launch_chain_t<SPEC_F32, true>(a, st) : launch_chain_t<SPEC_F32, false>(a, st);
}

}  // namespace sv
