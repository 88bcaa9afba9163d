// Pass-1 statistics and draw machinery shared by the chain and the stochastic
// tree verify (included by chain.cu and tree_sampled.cu; everything is
// inline or a template, so each translation unit holds its own copy).
//
// Pass 1, chain_rowstats_kernel: one short-lived CTA per 32 KB slice of a
// logit row (a.rows rows per request, request-major); it publishes its
// softmax statistics (M, S) as one nonzero 64-bit word, no fence, no wait.
// The draw: draw weights of 256-token chunks summed in 64-bit fixed point
// (chunk_sums), then the request's last CTA locates u*Z among the chunk sums
// and scans the one chunk that holds it (draw_token).  A TokenMask forces the
// weights of a few tokens to 0 (the stochastic tree's rejected children); a
// CutMask reads the tokens below each row's filter cut as -inf.
#pragma once

#include "kernels.cuh"

namespace sv {

namespace {

// Tokens whose draw weight is 0 (in shared memory); n == 0: none.
struct TokenMask {
  const int* tok;
  int n;
};

// Filtered rows (the wide filter): token t of the target row counts only
// when make_key(x_t, t) >= kp, of the draft row when >= kq; the others are
// read as logit -inf on that side.
struct CutMask {
  unsigned long long kp, kq;
};

// A bf16 pair (tokens t, t + 1) with the halves below the cut set to -inf.
__device__ __forceinline__ uint32_t cut_pair(uint32_t w, long t, unsigned long long k) {
  uint32_t r = w;
  if (make_key(__uint_as_float(w << 16), t) < k) r = (r & 0xffff0000u) | 0xff80u;
  if (make_key(__uint_as_float(w & 0xffff0000u), t + 1) < k) r = (r & 0x0000ffffu) | 0xff800000u;
  return r;
}

// Zeroes the weights of the masked tokens among t0 .. t0 + 7.
__device__ __forceinline__ void apply_mask(const TokenMask& m, long t0, float (&wv)[8]) {
  unsigned bits = 0;
  for (int i = 0; i < m.n; ++i) {
    const unsigned long long d = (unsigned long long)((long)m.tok[i] - t0);
    if (d < 8ull) bits |= 1u << (unsigned)d;
  }
  if (bits) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if ((bits >> i) & 1u) wv[i] = 0.f;
  }
}

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
    // here ch = (c, c) and nm = (-M c, -M c) rounded (see fma_offset):
    // 2^(x c - M c) with one packed fma per pair
    float2 e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 y = fma2(make_float2(bf16_lo(w[j]), bf16_hi(w[j])), ch, nm);
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
  b = rr / a.rows;
  r = rr - b * a.rows;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 6) chain_rowstats_kernel(const ChainArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // launched by launch_first
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
  constexpr bool kFma = VEC && DT == SPEC_BF16;
  float eps = 0.f;  // bf16: the rounding error of -Ms * c, restored in the sum below
  const float nmc = kFma ? fma_offset(Ms, a.c_rn, &eps) : -Ms;
  const float2 nm = make_float2(nmc, nmc),
               ch = kFma ? make_float2(a.c_rn, a.c_rn) : make_float2(a.c_hi, a.c_hi),
               cl = make_float2(a.c_lo, a.c_lo);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u)
    if (vbeg + tid + u * kThreads < vend) acc = add2(acc, vec_expsum<DT, VEC>(w[u], nm, ch, cl));
  float ssum = warp_sum(acc.x + acc.y);
  if (kFma) ssum *= ex2(eps);
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
    st_relaxed_u64(a.ws.stats + ((size_t)b * a.rows + r) * a.nsplit + s, stats_pack(M, S));
  }
}

// ------------------------------------------------------------------ pass 2
// The 8 draw weights of lane `lane` in chunk `c` (0 past the row's end):
// residual: 2^(c(xp - mp)) - lam * 2^(c(xq - mq)) clamped at 0, lam = Sp/Sq
// (that is Sp * max(0, p - q)); bonus (qrow == nullptr): 2^(c(xp - mp)).
template <int DT, bool VEC, bool MASK = false, bool CUT = false>
__device__ __forceinline__ void chunk_weights(const char* prow, const char* qrow, int c, int lane,
                                              int V, float mp, float mq, float lam, float c_hi,
                                              float c_lo, float c_rn, float (&wv)[8],
                                              TokenMask mask = TokenMask{nullptr, 0},
                                              CutMask cut = CutMask{0, 0}) {
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
  if constexpr (CUT) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (make_key(xp[i], t0 + i) < cut.kp) xp[i] = -INFINITY;
      if (qrow && make_key(xq[i], t0 + i) < cut.kq) xq[i] = -INFINITY;
    }
  }
  if constexpr (VEC && DT == SPEC_BF16) {
    // the one-fma exponents of chunk_sums' bf16 path, operation for operation
    float ep_, eq_ = 0.f;
    const float op = fma_offset(mp, c_rn, &ep_), oq = qrow ? fma_offset(mq, c_rn, &eq_) : 0.f;
    const float lam2 = qrow ? lam * ex2(eq_ - ep_) : 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 yp = fma2(make_float2(xp[2 * j], xp[2 * j + 1]), make_float2(c_rn, c_rn), make_float2(op, op));
      const float2 e_p = make_float2(ex2(yp.x), ex2(yp.y));
      if (qrow) {
        const float2 yq = fma2(make_float2(xq[2 * j], xq[2 * j + 1]), make_float2(c_rn, c_rn), make_float2(oq, oq));
        const float2 e_q = make_float2(ex2(yq.x), ex2(yq.y));
        const float2 w = fma2(make_float2(-lam2, -lam2), e_q, e_p);
        wv[2 * j] = fmaxf(w.x, 0.f);
        wv[2 * j + 1] = fmaxf(w.y, 0.f);
      } else {
        wv[2 * j] = e_p.x;
        wv[2 * j + 1] = e_p.y;
      }
    }
  } else {
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
  if constexpr (MASK) apply_mask(mask, t0, wv);
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
    const float2 yp = fma2(make_float2(bf16_lo(P[j]), bf16_hi(P[j])), ch, nmp);
    const float2 ep = make_float2(ex2(yp.x), ex2(yp.y));
    if (resid) {
      const float2 yq = fma2(make_float2(bf16_lo(Q[j]), bf16_hi(Q[j])), ch, nmq);
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
template <int DT, bool VEC, bool MASK = false, bool CUT = false>
__device__ __forceinline__ unsigned long long chunk_sums(const ChainArgs& a, const char* prow,
                                                         const char* qrow, int c0, int c1, float mp,
                                                         float mq, float lam,
                                                         unsigned long long* out,
                                                         TokenMask mask = TokenMask{nullptr, 0},
                                                         CutMask cut = CutMask{0, 0}) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long wtot = 0;
  if constexpr (VEC && DT == SPEC_BF16) {
    constexpr int GRP = 4;
    const bool resid = qrow != nullptr;
    // 2^(x c - m c) with one packed fma per pair, the offsets -m c rounded;
    // their rounding errors are a common factor of each side's weights, so
    // only their difference enters, through lam (the p side's factor is
    // common to every weight and leaves the draw unchanged)
    float ep_, eq_ = 0.f;
    const float op = fma_offset(mp, a.c_rn, &ep_), oq = resid ? fma_offset(mq, a.c_rn, &eq_) : 0.f;
    const float lam2 = resid ? lam * ex2(eq_ - ep_) : 0.f;
    const float2 nmp = make_float2(op, op), nmq = make_float2(oq, oq),
                 nlam = make_float2(-lam2, -lam2), ch = make_float2(a.c_rn, a.c_rn),
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
        if constexpr (CUT) {
          const long t = (long)c * kChunk + lane * 8;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            P[i][e] = cut_pair(P[i][e], t + 2 * e, cut.kp);
            if (resid) Q[i][e] = cut_pair(Q[i][e], t + 2 * e, cut.kq);
          }
        }
        float wv[8];
        weights8_bf16(P[i], Q[i], resid, nmp, nmq, nlam, ch, cl, wv);
        if constexpr (MASK) apply_mask(mask, (long)c * kChunk + lane * 8, wv);
        const unsigned long long f = to_fixed(warp_sum(tree8(wv)));
        if (lane == 0) out[c] = f;
        wtot += f;
      }
    }
  } else {
    for (int c = c0 + warp; c < c1; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC, MASK, CUT>(prow, qrow, c, lane, a.V, mp, mq, lam, a.c_hi, a.c_lo, a.c_rn, wv,
                                        mask, cut);
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
template <int DT, bool VEC, bool MASK = false, bool CUT = false>
__device__ int draw_token(const ChainArgs& a, int b, const char* prow, const char* qrow,
                          float mp, float mq, float lam, double u,
                          TokenMask mask = TokenMask{nullptr, 0}, CutMask cut = CutMask{0, 0}) {
  __shared__ unsigned long long sTarget, sPre, sZ;
  __shared__ unsigned long long sWarpTot[kWarps];
  __shared__ int sChunk, sTok, sRetry, sLastPos;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.nchunks, ni = a.nsplit2;
  unsigned long long* chunks = a.ws.chunks + (size_t)b * n;
  unsigned long long* items = a.ws.items + (size_t)b * ni;
  bool use_mask = MASK;  // cleared when the draw falls back to the unmasked row
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
      if (sChunk < 0) {  // (uniform: read after the loop's last barrier)
        if (tid == 0) {  // not reached while u < 1: the last positive chunk
          const int c = sLastPos < 0 ? 0 : sLastPos;
          sChunk = c;
          sPre = sZ - __ldcg(chunks + c);
        }
        __syncthreads();
      }
      break;
    }
    // The residual vanished numerically: draw from p_j instead (this CTA
    // recomputes every chunk and item sum; a rare path; without the token
    // mask, with the row's filter cut).
    qrow = nullptr;
    lam = 0.f;
    use_mask = false;
    for (int c = warp; c < n; c += kWarps) {
      float wv[8];
      chunk_weights<DT, VEC, false, CUT>(prow, nullptr, c, lane, a.V, mp, 0.f, 0.f, a.c_hi, a.c_lo, a.c_rn,
                                         wv, TokenMask{nullptr, 0}, cut);
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
  if (sChunk < 0) {  // (uniform) Z stayed 0 after the retry (not reached): chunk 0
    if (tid == 0) {
      sChunk = 0;
      sPre = 0;
    }
    __syncthreads();
  }
  if (warp == 0) {
    const int c = sChunk;
    float wv[8];
    if (use_mask)
      chunk_weights<DT, VEC, MASK, CUT>(prow, qrow, c, lane, a.V, mp, mq, lam, a.c_hi, a.c_lo, a.c_rn, wv,
                                        mask, cut);
    else
      chunk_weights<DT, VEC, false, CUT>(prow, qrow, c, lane, a.V, mp, mq, lam, a.c_hi, a.c_lo, a.c_rn, wv,
                                         TokenMask{nullptr, 0}, cut);
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

}  // namespace

}  // namespace sv
