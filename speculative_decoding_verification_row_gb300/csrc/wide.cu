// Filtered chain verify for kept sets of any size: top-p or min_p without
// top-k, and top-k above SPEC_MAX_TOPK (TensorRT-LLM walkthrough, rejection-
// sampling section: target and draft rows are filtered alike by temperature,
// top-k, top-p and min_p, in that order; vLLM anatomy page, "Speculative
// Decoding": accept/reject and the residual draw, here on the filtered
// rows).  filter.cu keeps explicit lists for top_k <= SPEC_MAX_TOPK.
//
// A kept set is a prefix of its row in (logit descending, token ascending)
// order, possibly shortened by min_p (a cut on the logit alone), so one
// 64-bit order key fixes it: token t is kept iff make_key(x_t, t) >= kcut.
// Each token's mass is e_t = 2^(c (x_t - M)) (c = log2(e)/T, M the row
// maximum).  Masses that decide a cut are summed in 2^-40 fixed point, so
// those sums are exact whatever their order; a row's total mass comes from
// pass 1's slice sums (fp32, about 1e-7 relative, far inside the oracle's
// 1e-6 near-tie window on the top-p cut).  Up to six stream-ordered grids
// (five when each row has one histogram CTA, four for min_p alone), each a
// programmatic dependent that waits for its predecessor before reading (no
// polling):
//   1. chain_rowstats_kernel (the chain's pass 1): the slice maxima and sums.
//   2. wide_hist_kernel, one CTA per 1 to 8 32 KB slices of a row (as many
//      as keep the grid at a full wave or more).  Only the heavy tokens,
//      those above a light depth, are binned: bin floor(32 c (M - x)) (2048
//      bins of 1/32 log2 unit), exact mass (and count when top-k cuts).  The
//      depth comes from a sample of the slice (an eighth): where the row's
//      tail below is estimated at half of (1 - top_p) Z, or where the count
//      above is estimated at 3 top_k + 256; on the headline shape about 3 %
//      of the tokens are heavy.  A 16-byte vector whose largest logit lies
//      below the depth (and below min_p's) is passed over after one packed
//      compare; the others are queued per warp and their tokens binned one
//      per lane.  The same pass sums min_p's mass and key.  min_p alone
//      needs no bins.
//   3. the bins step (bins_step): by the histogram CTA itself when it holds
//      the whole row, else by wide_bins_kernel, one CTA per row.  The row's
//      total mass is pass 1's (never below the heavy tokens' exact sum: the
//      light ones are the rest).  It checks exactly that the cut lies among
//      the bins every CTA filled (the top-k count or the top-p threshold is
//      reached above the shallowest depth) and otherwise rebuilds the row's
//      histogram with the a-priori depth D0 = log2(V / ((1 - top_p) Z)) + 1
//      (the V tokens below it weigh at most (1 - top_p) Z / 2) or, for
//      top-k, every token counted (and, should the cut still lie deeper --
//      top_p within pass 1's rounding of 1 -- every token binned, the total
//      then exact).  Then prefix sums give the bin where the top-k count is
//      reached and the range of bins the top-p threshold can fall in (the
//      top-k mass is known to within the top-k bin); the bins are rewritten
//      as their exclusive prefix sums.
//   4. wide_cand_kernel, one CTA per slice: the tokens of those bins (as
//      logit intervals, slightly widened) are listed per row (most rows:
//      tens to hundreds).
//   5. wide_cut_kernel, one CTA per row: exact selection over the listed
//      tokens' keys, with exact counts and masses (lists up to 512 ranked in
//      one pass, longer ones radix-selected eight bits at a time, a row with
//      more than 4096 rescanning itself): the top-k cut and its mass, then
//      the first token at which the running top-p mass reaches top_p times
//      it; min_p replaces the cut when its logit cut lies above.  Writes the
//      row's cut and kept mass.
//   6. wide_draw_kernel: the chain's draw items with the accept test on
//      p'(x_i) / q'(x_i) and the residual max(0, p' - q') (or the bonus p')
//      over the filtered rows: tokens below a row's cut read as -inf.
// Every call leaves the histograms, candidate lists, row records and
// statistics words zero, as the chain path does (a later call's layout may
// place its statistics words there).
#include <algorithm>
#include <mutex>

#include "draw.cuh"

namespace sv {

namespace {

constexpr int kStage = 2048;  // listed candidates the cut kernel stages in shared memory

__device__ __forceinline__ int mass_bin(float x, float M, float cR) {
  const float f = (M - x) * cR;  // >= 0; +inf for x = -inf
  return f < (float)kWideBins ? (int)f : kWideBins - 1;
}
// e = 2^(c (x - M)) <= 1 as an integer number of 2^-40.
__device__ __forceinline__ unsigned long long mass_fix(float x, float M, float c_hi, float c_lo) {
  return to_fixed(ex2(scaled(x - M, c_hi, c_lo)) * 256.f);
}

// The row's maximum and softmax sum (relative to it) from its slices'
// pass-1 words (all written by now); every CTA of the row gets the same.
__device__ float row_stats(const ChainArgs& a, int rr, float* Z) {
  __shared__ float s_m[kWarps], s_s[kWarps];
  const int tid = threadIdx.x;
  const unsigned long long* sw = a.ws.stats + (size_t)rr * a.nsplit;
  float m = -INFINITY;
  for (int u = tid; u < a.nsplit; u += kThreads) m = fmaxf(m, stats_unpack(ld_relaxed_u64(sw + u)).x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) s_m[tid >> 5] = m;
  __syncthreads();
  float M = s_m[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) M = fmaxf(M, s_m[i]);
  float sum = 0.f;
  if (M != -INFINITY)
    for (int u = tid; u < a.nsplit; u += kThreads) {
      const float2 e = stats_unpack(ld_relaxed_u64(sw + u));
      if (e.y > 0.f) sum += e.y * ex2(scaled(e.x - M, a.c_hi, a.c_lo));
    }
  sum = warp_sum(sum);
  if ((tid & 31) == 0) s_s[tid >> 5] = sum;
  __syncthreads();
  float S = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) S += s_s[i];
  *Z = S;
  return M == -INFINITY ? 0.f : M;
}

// A token's bin with the row's light tokens (bins >= b0) in the last bin.
__device__ __forceinline__ int wide_bin(float x, float M, float cR, int b0) {
  const int b = mass_bin(x, M, cR);
  return b < b0 ? b : kWideBins - 1;
}

// Block-wide exclusive prefix sum of one value per thread (thread order);
// *total receives the sum.
__device__ unsigned long long block_excl_u64(unsigned long long v, unsigned long long* total) {
  __shared__ unsigned long long s_w[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned long long incl = warp_incl_u64(v);
  if (lane == 31) s_w[warp] = incl;
  __syncthreads();
  unsigned long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    base += w < warp ? s_w[w] : 0;
    tot += s_w[w];
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

// The top-p threshold over a top-k mass Z: the running mass must reach
// top_p * Z, i.e. ceil(top_p * Z) in fixed point (at least 1).
__device__ __forceinline__ unsigned long long top_p_threshold(float top_p, unsigned long long Z) {
  const double t = ceil((double)top_p * (double)Z);
  return t < 1.0 ? 1ull : (unsigned long long)t;
}

// ------------------------------------------------------------------ 2
constexpr int kQueue = 64;   // queued vectors a warp holds before binning them
constexpr int kHistSlices = 8;  // 32 KB slices per histogram CTA, at most
constexpr int kLevels = 64;  // the sample's depth levels, half a log2 unit each

// The light depth that bounds the mass below it a priori: the V tokens
// deeper than D0 = log2(V / ((1 - top_p) Z)) + 1 weigh at most V 2^-D0 =
// (1 - top_p) Z / 2, so the top-p cut cannot fall among them (as a bin
// index, bins of 1/32 log2 unit).
__device__ __forceinline__ int safe_depth_bin(const ChainArgs& a, float Zs) {
  const float D0 = log2f((float)a.V / ((1.f - a.top_p) * fmaxf(Zs, 1.f))) + 1.f;
  const float fb = ceilf(D0 * (float)kWideBinsPerLog2) + 1.f;
  return fb < 1.f ? 1 : (fb >= (float)(kWideBins - 1) ? kWideBins - 1 : (int)fb);
}

// t moved down by a relative 1e-5 (and 1e-5 absolute): far more than the
// rounding of the logit-domain tests below.
__device__ __forceinline__ float widen_down(float t, float M) {
  return t - 1e-5f * (fabsf(M) + fabsf(t)) - 1e-5f;
}

struct HistParams {
  float M, c_hi, c_lo, cR;  // row maximum, log2(e)/T in two parts, bins per unit of logit
  float xthr;               // vectors whose largest logit is below xthr hold only light tokens
  float fb1;                // a token with (M - x) cR < fb1 is heavy
  float min_p;
  bool all;                 // every token is heavy (counted and binned)
};

// Heavy tokens are those of bins < b1 (all of them when b1 = kWideBins);
// xthr lies below every heavy token's logit and below every logit with
// 2^(c (x - M)) >= min_p (MINP).
__device__ __forceinline__ HistParams hist_params(const ChainArgs& a, float M, int b1, bool bins, bool minp) {
  HistParams h;
  h.M = M;
  h.c_hi = a.c_hi;
  h.c_lo = a.c_lo;
  h.cR = a.c_rn * (float)kWideBinsPerLog2;
  h.all = b1 >= kWideBins;
  h.fb1 = (float)b1;
  h.min_p = a.min_p;
  float x = INFINITY;
  if (bins) x = h.all ? -INFINITY : widen_down(M - (float)b1 / h.cR, M);
  if (minp) x = fminf(x, widen_down(M + log2f(a.min_p) / a.c_rn, M));
  h.xthr = x;
  return h;
}

// Where heavy tokens go: the CTA's shared histogram (three 14-bit parts of
// the 2^-40 fixed point in 32-bit adds; at most 2^17 tokens -- kHistSlices
// slices -- reach it between two flushes, so each part's sum stays below
// 2^31) ...
template <bool COUNT>
struct SharedBins {
  unsigned (*hm)[kWideBins];
  unsigned* hc;
  __device__ __forceinline__ void add(unsigned bin, float e) const {
    const unsigned long long f = to_fixed(e * 256.f);  // <= 2^40
    if (f) {
      atomicAdd(&hm[0][bin], (unsigned)f & 0x3fffu);
      atomicAdd(&hm[1][bin], (unsigned)(f >> 14) & 0x3fffu);
      atomicAdd(&hm[2][bin], (unsigned)(f >> 28));
    }
    if (COUNT) atomicAdd(&hc[bin], 1u);
  }
};
// ... or, when one CTA rebuilds a whole row, the row's global bins.
template <bool COUNT>
struct GlobalBins {
  unsigned long long* gh;
  unsigned* gc;
  __device__ __forceinline__ void add(unsigned bin, float e) const {
    const unsigned long long f = to_fixed(e * 256.f);
    if (f) atomicAdd(gh + bin, f);
    if (COUNT) atomicAdd(gc + bin, 1u);
  }
};

// One slice, held in registers (this thread's vectors v0 + u kThreads), into
// the bins.  A vector whose largest logit is below xthr holds only light
// tokens and is passed over (their mass is the row's total, from pass 1,
// less the heavy tokens').  Every other vector is queued by its warp
// (ballot); its tokens are then tested one per lane (4 vectors of 8 bf16 per
// step) and those at or above xthr queued again, so that the exact work --
// a heavy token's mass (and count) into its bin, and min_p's sum and key
// for every token with e >= min_p (MINP) -- runs 32 tokens at a time.
// Whatever xthr is, each token's bin is what its own test gives; xthr only
// decides how many tokens are tested one by one.
template <int DT, bool VEC, bool MINP, bool BINS, class Sink>
__device__ __forceinline__ void hist_slice(const Sink& sink, uint4* q, float* hq,
                                           const uint32_t (&w)[kVecPerThread][Io<DT, VEC>::NW], int v0,
                                           int vend, const HistParams& h, unsigned long long& zmin,
                                           unsigned& kinv) {
  using IO = Io<DT, VEC>;
  constexpr int EPV = IO::EPV;
  constexpr int VPS = 32 / EPV;  // queued vectors per warp step
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int hn = 0;  // tokens in hq (warp-uniform, < 32 between steps)
  auto take = [&](int n) {  // the first n <= 32 tokens of hq, one per lane
    __syncwarp();
    if (lane < n) {
      const float x = hq[lane];
      const float e = ex2(scaled(x - h.M, h.c_hi, h.c_lo));
      if constexpr (MINP) {
        if (e >= h.min_p) {
          zmin += to_fixed(e * 256.f);
          kinv = max(kinv, ~ord32(x));
        }
      }
      if constexpr (BINS) {
        const float fbin = (h.M - x) * h.cR;
        if (h.all || fbin < h.fb1) sink.add((unsigned)(int)fminf(fbin, (float)(kWideBins - 1)), e);
      }
    }
    __syncwarp();
  };
  auto drain = [&](int qn) {
    __syncwarp();
    for (int q0 = 0; q0 < qn; q0 += VPS) {
      const int qi = q0 + lane / EPV, el = lane % EPV;
      float x = -INFINITY;
      if (qi < qn) {
        if constexpr (VEC && DT == SPEC_BF16)
          x = __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(q + qi)[el] << 16);
        else if constexpr (VEC)
          x = reinterpret_cast<const float*>(q + qi)[el];
        else
          x = __uint_as_float(q[qi].x);  // (scalar bf16 is held in the high half)
      }
      // every token of a queued vector when all are heavy (-inf included)
      const bool need = qi < qn && (h.all || x >= h.xthr);
      const unsigned m = __ballot_sync(0xffffffffu, need);
      if (need) hq[hn + __popc(m & below)] = x;
      hn += __popc(m);
      if (hn >= 32) {
        take(32);
        if (lane < hn - 32) hq[lane] = hq[32 + lane];
        __syncwarp();
        hn -= 32;
      }
    }
    __syncwarp();
  };
  int qn = 0;  // warp-uniform
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const bool fl = v0 + u * kThreads < vend && IO::vmax(w[u]) >= h.xthr;
    const unsigned m = __ballot_sync(0xffffffffu, fl);
    if (fl) {
      uint4 v;
      v.x = w[u][0];
      if constexpr (IO::NW == 4) {
        v.y = w[u][1];
        v.z = w[u][2];
        v.w = w[u][3];
      } else {
        v.y = v.z = v.w = 0u;
      }
      q[qn + __popc(m & below)] = v;
    }
    qn += __popc(m);
    if (qn > kQueue - 32) {
      drain(qn);
      qn = 0;
    }
  }
  if (qn) drain(qn);
  if (hn) take(hn);
}

// This slice's light depth (a bin index): from a sample of the slice, its
// first vector per thread (an eighth of it), the shallowest depth, in half
// log2 units, at which the row's estimated mass below stays under half of
// (1 - top_p) Z with at least 16 sampled tokens above it (top-p: a tail
// estimate resting on fewer tokens is not trusted), or the estimated count
// above reaches 3 top_k + 256 (top-k); never deeper than b0.  Only a speed choice: the bins grid checks
// exactly that the row's cut lies above the row's shallowest light depth
// and rebuilds the row otherwise.
template <int DT, bool VEC, bool COUNT>
__device__ int sample_depth(const uint32_t (&w0)[Io<DT, VEC>::NW], bool valid, const ChainArgs& a, float M,
                            float Zs, int b0, float* lm, unsigned* lc, float* zsub, unsigned* nsub, int* b1out) {
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lmax = COUNT ? kLevels : min(kLevels, b0 / 16);
  float zs = 0.f;
  if (valid) {
    float x[IO::EPV];
    IO::unpack(w0, x);
    const float c2 = 2.f * a.c_rn;
#pragma unroll
    for (int i = 0; i < IO::EPV; ++i) {
      const float dl = (M - x[i]) * c2;  // depth in half log2 units (+inf for -inf)
      const int lv = dl < (float)lmax ? (int)dl : lmax;
      if (lv < lmax) atomicAdd(lc + lv, 1u);
      if (!COUNT) {
        const float e = ex2(-0.5f * dl);
        zs += e;
        if (lv < lmax) atomicAdd(lm + lv, e);
      }
    }
  }
  unsigned ns = valid ? (unsigned)IO::EPV : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    zs += __shfl_xor_sync(0xffffffffu, zs, o);
    ns += __shfl_xor_sync(0xffffffffu, ns, o);
  }
  if (lane == 0) {
    if (!COUNT) atomicAdd(zsub, zs);
    atomicAdd(nsub, ns);
  }
  __syncthreads();
  if (warp == 0) {
    const float scale = *nsub ? (float)a.V / (float)*nsub : 0.f;
    const int j0 = 2 * lane, j1 = j0 + 1;
    // running totals over the levels above j0 and j1 (lane order = depth
    // order): sampled tokens, and (top-p) their mass
    const float n0 = (float)lc[j0], n1 = (float)lc[j1];
    const float v0 = COUNT ? 0.f : lm[j0], v1 = COUNT ? 0.f : lm[j1];
    float ninc = n0 + n1, inc = v0 + v1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, ninc, o), t2 = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) {
        ninc += t;
        inc += t2;
      }
    }
    const float nab0 = ninc - n0 - n1, nab1 = nab0 + n0;
    const float above0 = inc - v0 - v1, above1 = above0 + v0;
    bool ok0, ok1;
    if (COUNT) {  // tokens above the depth
      const float need = 3.f * (float)a.top_k + 256.f;
      ok0 = j0 >= 1 && scale * nab0 >= need;
      ok1 = scale * nab1 >= need;
    } else {  // mass below the depth
      const float tail = 0.5f * (1.f - a.top_p) * Zs, z = *zsub;
      ok0 = j0 >= 1 && j0 <= lmax && nab0 >= 16.f && scale * (z - above0) <= tail;
      ok1 = j1 <= lmax && nab1 >= 16.f && scale * (z - above1) <= tail;
    }
    const unsigned m0 = __ballot_sync(0xffffffffu, ok0), m1 = __ballot_sync(0xffffffffu, ok1);
    int j = kLevels;
    if (m0) j = 2 * (__ffs(m0) - 1);
    if (m1) j = min(j, 2 * (__ffs(m1) - 1) + 1);
    if (lane == 0) *b1out = j < kLevels ? min(16 * j, b0) : b0;
  }
  __syncthreads();
  return *b1out;
}

// Bins b of a row are held 8 per thread (thread t: 8t .. 8t + 7).
constexpr int kBinsPerThread = kWideBins / kThreads;
static_assert(kBinsPerThread * kThreads == kWideBins, "bins per thread");

// The bins step of one row, by one CTA.  load(m, c) gives this thread's
// bins 8 tid .. 8 tid + 7 (mass, count) as the histogram left them (bins
// below b1 complete, the deeper ones partial); rebuild(b) rebuilds the
// histogram with light depth b.  The row's total mass is pass 1's (Zs,
// never below the heavy tokens' exact sum; the light tokens' share of it is
// not binned) for top-p, the exact sum when every token is heavy (top-k, or
// b = kWideBins).  The cut must lie above b1: the bins above it must reach
// the top-k count (top-k) or the top-p threshold of the total (top-p alone);
// if not, the row is rebuilt with the a-priori depth (every token counted,
// for top-k), and, should top_p be within pass 1's rounding of 1, with every
// token binned.  Then the bins become their exclusive prefix sums (gh, gc:
// this thread's eight) and the row's record gets the top-k bin, the top-p
// bin range, the light depth and the total.
template <bool COUNT, class Load, class Rebuild>
__device__ __forceinline__ void bins_step(const ChainArgs& a, WideRow* wr, int b1, float Zs, const Load& load,
                                          const Rebuild& rebuild, unsigned long long* gh, unsigned* gc) {
  __shared__ int s_bk, s_blo, s_bhi;
  __shared__ unsigned long long s_mb, s_mbin;
  const int tid = threadIdx.x;
  const bool count_cut = COUNT && a.top_k < a.V;
  unsigned long long m[kBinsPerThread];
  unsigned c[kBinsPerThread];
  unsigned long long Z = 0, C = 0, NC = 0;
  auto gather = [&]() {  // the bins, the heavy total, the complete region's mass (count)
    load(m, c);
    unsigned long long tm = 0, cm = 0, cc = 0;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      tm += m[j];
      if (kBinsPerThread * tid + j < b1) {
        cm += m[j];
        cc += c[j];
      }
    }
    unsigned long long zh;
    block_excl_u64(tm, &zh);
    block_excl_u64(cm, &C);
    if (count_cut) block_excl_u64(cc, &NC);
    Z = COUNT || b1 >= kWideBins ? zh : max(zh, to_fixed(Zs * 256.f));  // (every token heavy: exact)
  };
  auto cut_above = [&]() {  // (an empty row has no cut)
    return b1 >= kWideBins || Z == 0 ||
           (count_cut ? NC >= (unsigned long long)a.top_k : C >= top_p_threshold(a.top_p, Z));
  };
  gather();
  if (!cut_above()) {  // (uniform)
    b1 = COUNT ? kWideBins : safe_depth_bin(a, Zs);
    rebuild(b1);
    gather();
    if (!cut_above()) {
      b1 = kWideBins;
      rebuild(b1);
      gather();
    }
  }
  if (b1 < kWideBins) {  // the bins from b1 on merge into the last bin
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      const int bin = kBinsPerThread * tid + j;
      if (bin >= b1) {
        m[j] = bin == kWideBins - 1 ? Z - C : 0;
        c[j] = 0;
      }
    }
  }
  if (tid == 0) {
    s_bk = s_blo = s_bhi = -1;
    s_mb = 0;
    s_mbin = 0;
  }
  unsigned long long tm = 0, tc = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    tm += m[j];
    tc += c[j];
  }
  unsigned long long N;
  const unsigned long long pm = block_excl_u64(tm, &Z);
  const unsigned long long pc = COUNT ? block_excl_u64(tc, &N) : 0;
  // top-k: the bin where the running count reaches top_k
  if (count_cut) {
    unsigned long long cb = pc, mb = pm;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      if (cb < (unsigned long long)a.top_k && (unsigned long long)a.top_k <= cb + c[j]) {
        s_bk = kBinsPerThread * tid + j;
        s_mb = mb;
        s_mbin = m[j];
      }
      cb += c[j];
      mb += m[j];
    }
  }
  __syncthreads();
  if (a.top_p < 1.f) {
    // the top-k mass lies in [zlo, zhi]; so does the threshold's bin range
    const unsigned long long zlo = s_bk >= 0 ? s_mb : Z, zhi = s_bk >= 0 ? s_mb + s_mbin : Z;
    const unsigned long long tl = top_p_threshold(a.top_p, zlo), th = top_p_threshold(a.top_p, zhi);
    unsigned long long mb = pm;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      if (mb < tl && tl <= mb + m[j]) s_blo = kBinsPerThread * tid + j;
      if (mb < th && th <= mb + m[j]) s_bhi = kBinsPerThread * tid + j;
      mb += m[j];
    }
  }
  // The bins become their exclusive prefix sums (mass, and count when top-k
  // cuts): the cut kernel reads the few it needs.
  {
    unsigned long long mb = pm, cb = pc;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      gh[j] = mb;
      if (COUNT) gc[j] = (unsigned)cb;
      mb += m[j];
      cb += c[j];
    }
  }
  __syncthreads();
  if (tid == 0) {
    wr->bk = s_bk;
    wr->blo = s_blo;
    wr->bhi = s_blo >= 0 ? s_bhi : -1;
    wr->b0 = b1;  // from here on: the row's light depth
    wr->ztot = Z;
  }
}

// BINS = false (min_p alone): no histogram, only the min_p mass and key.
// COUNT: top-k cuts (every token counted and binned when top_k >= V).
template <int DT, bool VEC, bool COUNT, bool MINP, bool BINS>
__global__ void __launch_bounds__(kThreads, 4) wide_hist_kernel(const ChainArgs a) {
  __shared__ unsigned hm[3][kWideBins];
  __shared__ unsigned hc[COUNT ? kWideBins : 1];
  __shared__ uint4 sq[kWarps][kQueue];
  __shared__ float shq[kWarps][64];
  __shared__ float s_lm[kLevels];
  __shared__ unsigned s_lc[kLevels];
  __shared__ float s_zsub;
  __shared__ unsigned s_nsub;
  __shared__ int s_b1;
  __shared__ unsigned long long s_z[kWarps];
  __shared__ unsigned s_k[kWarps];
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Each row's slices are split among `groups` CTAs (the grid's size over
  // the rows), spc consecutive slices each, taken in turn: the row
  // statistics, the sampled depth (from the first) and the shared bins serve
  // them all.
  const int groups = (int)(gridDim.x / ((unsigned)a.B * (unsigned)a.rows));
  const int spc = (a.nsplit + groups - 1) / groups;
  const int rr = blockIdx.x / groups, c = blockIdx.x - rr * groups;
  int b, r;
  slice_row(a, rr, b, r);
  if (BINS)
    for (int i = tid; i < kWideBins; i += kThreads) {
      hm[0][i] = hm[1][i] = hm[2][i] = 0u;
      if (COUNT) hc[i] = 0;
    }
  if (tid < kLevels) {
    s_lm[tid] = 0.f;
    s_lc[tid] = 0u;
  }
  if (tid == 0) {
    s_zsub = 0.f;
    s_nsub = 0u;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
  uint32_t w[kVecPerThread][IO::NW];
  auto load_slice = [&](int s) {
    const int vbeg = s * a.vps, vend = min(a.nvec, vbeg + a.vps);
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = vbeg + tid + u * kThreads;
      if (v < vend) {
        IO::load(row, v, w[u]);
      } else {  // past the row: -inf (no mass; never queued)
#pragma unroll
        for (int q = 0; q < IO::NW; ++q) w[u][q] = (VEC && DT == SPEC_BF16) ? 0xff80ff80u : 0xff800000u;
      }
    }
  };
  const int s0 = c * spc;
  int vbeg = s0 * a.vps, vend = min(a.nvec, vbeg + a.vps);
  load_slice(s0);
  float Zs;
  const float M = row_stats(a, rr, &Zs);  // also orders the clearing above before the adds
  const bool count_active = COUNT && a.top_k < a.V;  // (else every token is counted)
  int b1 = kWideBins;
  if constexpr (BINS) {
    const int b0 = COUNT ? kWideBins : safe_depth_bin(a, Zs);
    b1 = COUNT && !count_active
             ? kWideBins
             : sample_depth<DT, VEC, COUNT>(w[0], vbeg + tid < vend, a, M, Zs, b0, s_lm, s_lc, &s_zsub,
                                            &s_nsub, &s_b1);
  }
  WideRow* wr = a.ws.wrow + rr;
  if (tid == 0) {
    if (c == 0) wr->M = M;                          // every CTA of the row computes the same
    // The record's b0 holds kWideBins + 1 - (the smallest light depth of the
    // row's slices) until the bins grid replaces it with the row's depth.
    if (BINS) atomicMax(&wr->b0, kWideBins + 1 - b1);
  }
  const HistParams h = hist_params(a, M, b1, BINS, MINP);
  unsigned long long zmin = 0;
  unsigned kinv = 0;
  hist_slice<DT, VEC, MINP, BINS>(SharedBins<COUNT>{hm, hc}, sq[warp], shq[warp], w, vbeg + tid, vend, h, zmin,
                                  kinv);
  for (int s = s0 + 1; s < min(a.nsplit, s0 + spc); ++s) {  // (uniform) the others
    load_slice(s);
    vbeg = s * a.vps;
    vend = min(a.nvec, vbeg + a.vps);
    hist_slice<DT, VEC, MINP, BINS>(SharedBins<COUNT>{hm, hc}, sq[warp], shq[warp], w, vbeg + tid, vend, h,
                                    zmin, kinv);
  }
  if constexpr (BINS) {
    unsigned long long* gh = a.ws.whist + (size_t)rr * kWideBins;
    unsigned* gc = a.ws.wcount + (size_t)rr * kWideBins;
    __syncthreads();
    auto bin_mass = [&](int i) {
      return ((unsigned long long)hm[2][i] << 28) + ((unsigned long long)hm[1][i] << 14) + hm[0][i];
    };
    if (groups == 1) {
      // (uniform) The whole row is here: the bins step in place, from the
      // shared bins, a rebuild re-reading this CTA's slices into them.
      auto load = [&](unsigned long long (&m)[kBinsPerThread], unsigned (&cn)[kBinsPerThread]) {
#pragma unroll
        for (int j = 0; j < kBinsPerThread; ++j) {
          m[j] = bin_mass(kBinsPerThread * tid + j);
          cn[j] = COUNT ? hc[kBinsPerThread * tid + j] : 0u;
        }
      };
      auto rebuild = [&](int depth) {
        __syncthreads();  // every thread has read the bins
        for (int i = tid; i < kWideBins; i += kThreads) {
          hm[0][i] = hm[1][i] = hm[2][i] = 0u;
          if (COUNT) hc[i] = 0;
        }
        __syncthreads();
        const HistParams hb = hist_params(a, M, depth, true, false);
        for (int s = s0; s < min(a.nsplit, s0 + spc); ++s) {
          load_slice(s);
          const int vb = s * a.vps, ve = min(a.nvec, vb + a.vps);
          unsigned long long zd = 0;
          unsigned kd = 0;
          hist_slice<DT, VEC, false, true>(SharedBins<COUNT>{hm, hc}, sq[warp], shq[warp], w, vb + tid, ve, hb,
                                           zd, kd);
        }
        __syncthreads();
      };
      bins_step<COUNT>(a, wr, b1, Zs, load, rebuild, gh + kBinsPerThread * tid, gc + kBinsPerThread * tid);
    } else {
      for (int i = tid; i < min(b1, kWideBins); i += kThreads) {  // heavy bins lie below b1
        const unsigned long long m = bin_mass(i);
        if (m) atomicAdd(gh + i, m);
        if (COUNT && hc[i]) atomicAdd(gc + i, hc[i]);
      }
    }
  }
  if (MINP) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      zmin += __shfl_xor_sync(0xffffffffu, zmin, o);
      kinv = max(kinv, __shfl_xor_sync(0xffffffffu, kinv, o));
    }
    if (lane == 0) {
      s_z[warp] = zmin;
      s_k[warp] = kinv;
    }
    __syncthreads();
    if (tid == 0) {
      unsigned long long z = 0;
      unsigned kk = 0;
#pragma unroll
      for (int i = 0; i < kWarps; ++i) {
        z += s_z[i];
        kk = max(kk, s_k[i]);
      }
      if (z) atomicAdd(&wr->zmin, z);
      if (kk) atomicMax(&wr->kmin_inv, kk);
    }
  }
}

// ------------------------------------------------------------------ 3

// The row's histogram rebuilt by this one CTA with light depth b0 (every
// token heavy when b0 = kWideBins), its slices streaming through the
// registers in turn, straight into the row's global bins (cleared first).
template <int DT, bool VEC, bool COUNT>
__device__ void rebuild_row(const ChainArgs& a, int rr, float M, int b0, uint4* q, float* hq,
                            unsigned long long* gh, unsigned* gc) {
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x;
  int b, r;
  slice_row(a, rr, b, r);
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
  for (int i = tid; i < kWideBins; i += kThreads) {
    gh[i] = 0;
    if (COUNT) gc[i] = 0;
  }
  __syncthreads();
  const HistParams h = hist_params(a, M, b0, true, false);
  for (int s = 0; s < a.nsplit; ++s) {
    const int vbeg = s * a.vps;
    const int vend = min(a.nvec, vbeg + a.vps);
    uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
    for (int u = 0; u < kVecPerThread; ++u) {
      const int v = vbeg + tid + u * kThreads;
      if (v < vend) {
        IO::load(row, v, w[u]);
      } else {
#pragma unroll
        for (int k = 0; k < IO::NW; ++k) w[u][k] = (VEC && DT == SPEC_BF16) ? 0xff80ff80u : 0xff800000u;
      }
    }
    unsigned long long zd = 0;
    unsigned kd = 0;
    hist_slice<DT, VEC, false, true>(GlobalBins<COUNT>{gh, gc}, q, hq, w, vbeg + tid, vend, h, zd, kd);
  }
  __syncthreads();  // the adds above before the reads after
}

// Rows split over several histogram CTAs: the bins step on the row's global
// histogram, a rebuild streaming the row through this CTA.
template <int DT, bool VEC, bool COUNT>
__global__ void __launch_bounds__(kThreads, 4) wide_bins_kernel(const ChainArgs a) {
  __shared__ uint4 sq[kWarps][kQueue];
  __shared__ float shq[kWarps][64];
  const int tid = threadIdx.x;
  const int rr = blockIdx.x, b = rr / a.rows, r = rr - b * a.rows;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  unsigned long long* gh0 = a.ws.whist + (size_t)rr * kWideBins;
  unsigned* gc0 = a.ws.wcount + (size_t)rr * kWideBins;
  unsigned long long* gh = gh0 + kBinsPerThread * tid;
  unsigned* gc = gc0 + kBinsPerThread * tid;
  WideRow* wr = a.ws.wrow + rr;
  const int b1 = kWideBins + 1 - wr->b0;  // the row's shallowest slice depth (encoded by the slices)
  float Zs = 0.f;
  if (!COUNT) row_stats(a, rr, &Zs);
  auto load = [&](unsigned long long (&m)[kBinsPerThread], unsigned (&c)[kBinsPerThread]) {
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      m[j] = gh[j];
      c[j] = COUNT ? gc[j] : 0u;
    }
  };
  auto rebuild = [&](int depth) {
    rebuild_row<DT, VEC, COUNT>(a, rr, wr->M, depth, sq[tid >> 5], shq[tid >> 5], gh0, gc0);
  };
  bins_step<COUNT>(a, wr, b1, Zs, load, rebuild, gh, gc);
}

// ------------------------------------------------------------------ 4
// The bits of this thread's tokens whose logits lie in [lo1, hi1] (or
// [lo2, hi2] when TWO); v0 is its first vector.
template <int DT, bool VEC, bool TWO>
__device__ __forceinline__ unsigned long long listed_bits(const uint32_t (&w)[kVecPerThread][Io<DT, VEC>::NW],
                                                          int v0, int vend, float lo1, float hi1, float lo2,
                                                          float hi2) {
  using IO = Io<DT, VEC>;
  unsigned long long sel = 0;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    if (v0 + u * kThreads >= vend) continue;
    float x[IO::EPV];
    IO::unpack(w[u], x);
#pragma unroll
    for (int i = 0; i < IO::EPV; ++i) {
      bool in = x[i] >= lo1 && x[i] <= hi1;
      if (TWO) in = in || (x[i] >= lo2 && x[i] <= hi2);
      if (in) sel |= 1ull << (u * IO::EPV + i);
    }
  }
  return sel;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 5) wide_cand_kernel(const ChainArgs a) {
  __shared__ unsigned s_base;
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x;
  const int rr = blockIdx.x / a.nsplit, s = blockIdx.x - rr * a.nsplit;
  int b, r;
  slice_row(a, rr, b, r);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  const char* row = row_ptr(a, b, r, (size_t)a.V * IO::ES);
  const int vbeg = s * a.vps;
  const int vend = min(a.nvec, vbeg + a.vps);
  uint32_t w[kVecPerThread][IO::NW];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int v = vbeg + tid + u * kThreads;
    if (v < vend) IO::load(row, v, w[u]);
  }
  WideRow* wr = a.ws.wrow + rr;  // read while the slice is in flight
  const int bk = wr->bk, blo = wr->blo, bhi = wr->bhi;
  if (bk < 0 && blo < 0) return;  // no cut falls inside a bin: nothing to list
  const float M = wr->M;
  const int b0 = wr->b0;
  const float cR = a.c_rn * (float)kWideBinsPerLog2;
  // Bin b holds the tokens with (M - x) cR in [b, b + 1), and the last bin
  // everything from min(b0, kWideBins - 1) on (down to -inf).  The listed
  // bins as logit intervals [xlo, xhi], widened by a relative 1e-5 so that
  // they hold every token of those bins whatever the rounding; the cut
  // kernel keeps only the tokens whose bin is one it needs.
  auto lo_of = [&](int bin) { return bin == kWideBins - 1 ? (float)min(b0, kWideBins - 1) : (float)bin; };
  auto xhi_of = [&](float flo) {  // the largest logit of bins >= flo
    const float t = M - flo / cR;
    return t + 1e-5f * (fabsf(M) + fabsf(t)) + 1e-30f;
  };
  auto xlo_of = [&](int bin) {  // the smallest logit of bins <= bin
    if (bin == kWideBins - 1) return -INFINITY;
    const float t = M - (float)(bin + 1) / cR;
    return t - 1e-5f * (fabsf(M) + fabsf(t)) - 1e-30f;
  };
  const float k_hi = bk >= 0 ? xhi_of(lo_of(bk)) : -INFINITY, k_lo = bk >= 0 ? xlo_of(bk) : INFINITY;
  const float r_hi = blo >= 0 ? xhi_of(lo_of(blo)) : -INFINITY, r_lo = blo >= 0 ? xlo_of(bhi) : INFINITY;
  // bit u * EPV + i: element i of vector u is listed (one interval in the
  // usual cases: top-p alone or top-k alone)
  unsigned long long sel =
      bk >= 0 && blo >= 0
          ? listed_bits<DT, VEC, true>(w, vbeg + tid, vend, k_lo, k_hi, r_lo, r_hi)
          : (bk >= 0 ? listed_bits<DT, VEC, false>(w, vbeg + tid, vend, k_lo, k_hi, 0.f, 0.f)
                     : listed_bits<DT, VEC, false>(w, vbeg + tid, vend, r_lo, r_hi, 0.f, 0.f));
  unsigned long long total;
  const unsigned long long off = block_excl_u64((unsigned long long)__popcll(sel), &total);
  if (total == 0) return;  // uniform
  if (tid == 0) s_base = atomicAdd(&wr->ncand, (unsigned)total);
  __syncthreads();
  unsigned pos = s_base + (unsigned)off;
  unsigned* out = a.ws.wcand + (size_t)rr * kWideCandCap;
  while (sel) {
    const int bit = __ffsll((long long)sel) - 1;
    sel &= sel - 1;
    if (pos < (unsigned)kWideCandCap) {
      const int u = bit / IO::EPV, i = bit - u * IO::EPV;
      out[pos] = (unsigned)((vbeg + tid + u * kThreads) * IO::EPV + i);
    }
    ++pos;
  }
}

// ------------------------------------------------------------------ 5
struct SelSmem {
  unsigned cnt[256];
  unsigned long long mass[256];
  int digit;
  unsigned long long before_w, before_m;
};

// Among the row's listed tokens i < n that satisfy pred(key, bin), in
// decreasing key order (logit descending, token ascending), the first at
// which the running weight (a count, or the fixed-point mass when by_mass)
// reaches `target` (1 <= target <= their total): radix selection over the
// 64-bit keys, eight bits at a time from the top, with the exact weight of
// every digit.  Returns its key; *mass_incl receives the mass up to and
// including it.
template <class Get, class Pred>
__device__ unsigned long long radix_select(int n, const Get& get, const Pred& pred, bool by_mass,
                                           unsigned long long target, float M, const ChainArgs& a,
                                           SelSmem& S, unsigned long long* mass_incl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long prefix = 0, mbefore = 0;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += kThreads) {
      S.cnt[i] = 0;
      S.mass[i] = 0;
    }
    __syncthreads();
    const unsigned long long hi = shift == 56 ? 0ull : ~0ull << (shift + 8);
    for (int i = tid; i < n; i += kThreads) {
      unsigned long long K;
      int bin;
      get(i, K, bin);
      if (!pred(K, bin) || ((K ^ prefix) & hi)) continue;
      const int d = (int)(K >> shift) & 255;
      atomicAdd(&S.cnt[d], 1u);
      const unsigned long long f = mass_fix(unord32((uint32_t)(K >> 32)), M, a.c_hi, a.c_lo);
      if (f) atomicAdd(&S.mass[d], f);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l: digits 255 - 8l down to 248 - 8l (decreasing keys first)
      unsigned long long wv[8], mv[8], lw = 0, lm = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int d = 255 - 8 * lane - j;
        mv[j] = S.mass[d];
        wv[j] = by_mass ? mv[j] : (unsigned long long)S.cnt[d];
        lw += wv[j];
        lm += mv[j];
      }
      const unsigned long long iw = warp_incl_u64(lw), im = warp_incl_u64(lm);
      unsigned long long bw = iw - lw, bm = im - lm;
      if (bw < target && target <= iw) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (bw < target && target <= bw + wv[j]) {
            S.digit = 255 - 8 * lane - j;
            S.before_w = bw;
            S.before_m = bm;
          }
          bw += wv[j];
          bm += mv[j];
        }
      }
    }
    __syncthreads();
    prefix |= (unsigned long long)S.digit << shift;
    target -= S.before_w;
    mbefore += S.before_m;
    __syncthreads();
  }
  *mass_incl = mbefore + mass_fix(unord32((uint32_t)(prefix >> 32)), M, a.c_hi, a.c_lo);
  return prefix;
}

// Among the staged tokens i < n that satisfy pred(key, bin), in decreasing
// key order, the first at which the running weight (a count, or the mass
// when by_mass) reaches `target`: every thread ranks its own tokens against
// all n (O(n) each, one barrier), for short lists.  Returns the key; *mass_incl
// receives the mass up to and including it.
template <class Pred>
__device__ unsigned long long rank_select(int n, const unsigned long long* sKey, const unsigned short* sBin,
                                          const unsigned long long* sF, const Pred& pred, bool by_mass,
                                          unsigned long long target, unsigned long long* mass_incl) {
  __shared__ unsigned long long s_key, s_mass;
  for (int i = threadIdx.x; i < n; i += kThreads) {
    const unsigned long long K = sKey[i];
    if (!pred(K, sBin[i])) continue;
    unsigned long long bw = 0, bm = 0;
    for (int t = 0; t < n; ++t) {
      const unsigned long long Kt = sKey[t];
      if (Kt > K && pred(Kt, sBin[t])) {
        bm += sF[t];
        bw += by_mass ? sF[t] : 1ull;
      }
    }
    const unsigned long long w = by_mass ? sF[i] : 1ull;
    if (bw < target && target <= bw + w) {
      s_key = K;
      s_mass = bm + sF[i];
    }
  }
  __syncthreads();
  *mass_incl = s_mass;
  const unsigned long long K = s_key;
  __syncthreads();
  return K;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) wide_cut_kernel(const ChainArgs a) {
  constexpr int kMeStage = 256;  // prefix sums of the top-p bin range held at once
  __shared__ unsigned long long sKey[kStage], sF[kStage];
  __shared__ unsigned short sBin[kStage];
  __shared__ unsigned long long sMe[kMeStage + 1];
  __shared__ SelSmem S;
  __shared__ unsigned long long s_mek, s_cbk;
  __shared__ int s_bp;
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const int tid = threadIdx.x;
  const int rr = blockIdx.x, b = rr / a.rows, r = rr - b * a.rows;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  const char* row = row_ptr(a, b, r, (size_t)a.V * ES);
  WideRow* wr = a.ws.wrow + rr;
  const bool bins = a.top_k > 0 || a.top_p < 1.f;  // min_p alone has no histogram
  const int bk = bins ? wr->bk : -1, blo = bins ? wr->blo : -1, bhi = bins ? wr->bhi : -1, b0 = wr->b0;
  const unsigned ncand = wr->ncand;
  const unsigned long long zmin = wr->zmin, Z = wr->ztot;
  const unsigned kinv = wr->kmin_inv;
  const float M = wr->M;
  unsigned long long* gh = a.ws.whist + (size_t)rr * kWideBins;  // exclusive prefix sums now
  unsigned* gc = a.ws.wcount + (size_t)rr * kWideBins;
  const bool count_cut = a.top_k > 0;
  auto me = [&](int bin) { return bin >= kWideBins ? Z : gh[bin]; };
  if (tid == 0) {
    s_mek = bk >= 0 ? me(bk) : 0;
    s_cbk = bk >= 0 ? gc[bk] : 0;
  }
  // Stage the listed tokens (or, past the list's capacity, read the row).
  const bool listed = ncand <= (unsigned)kWideCandCap;
  const int n = listed ? (int)ncand : a.V;
  const bool staged = listed && n <= kStage;
  const unsigned* cand = a.ws.wcand + (size_t)rr * kWideCandCap;
  const float cR = a.c_rn * (float)kWideBinsPerLog2;
  if (staged)
    for (int i = tid; i < n; i += kThreads) {
      const unsigned t = cand[i];
      const float x = load_logit<DT>(row, t);
      sKey[i] = make_key(x, t);
      sBin[i] = (unsigned short)wide_bin(x, M, cR, b0);
      sF[i] = mass_fix(x, M, a.c_hi, a.c_lo);
    }
  __syncthreads();
  auto get = [&](int i, unsigned long long& K, int& bin) {
    if (staged) {
      K = sKey[i];
      bin = sBin[i];
    } else {
      const unsigned t = listed ? cand[i] : (unsigned)i;
      const float x = load_logit<DT>(row, t);
      K = make_key(x, t);
      bin = wide_bin(x, M, cR, b0);
    }
  };
  const bool short_list = staged && n <= 512;
  unsigned long long kcut = 0, kept = Z, zk = Z, kk = 0;
  bool ok = true;
  if (bk >= 0) {  // top-k: the (top_k - count above)-th token of bin bk
    unsigned long long in;
    auto pk = [&](unsigned long long, int bin) { return bin == bk; };
    const unsigned long long tk = (unsigned long long)a.top_k - s_cbk;
    kk = short_list ? rank_select(n, sKey, sBin, sF, pk, false, tk, &in)
                    : radix_select(n, get, pk, false, tk, M, a, S, &in);
    kcut = kk;
    zk = s_mek + in;
    kept = zk;
  }
  if (a.top_p < 1.f) {
    const unsigned long long th = top_p_threshold(a.top_p, zk);
    // the last bin (within the top-k set) whose preceding mass is below the
    // threshold: bk, or one of blo .. bhi (their prefixes staged in pieces)
    if (tid == 0) s_bp = -1;
    __syncthreads();
    const int hi = bk >= 0 ? min(bhi, bk) : bhi;
    for (int c0 = blo; c0 <= hi; c0 += kMeStage) {
      const int cnt = min(kMeStage, hi - c0 + 1);
      for (int i = tid; i <= cnt; i += kThreads) sMe[i] = me(c0 + i);
      __syncthreads();
      for (int i = tid; i < cnt; i += kThreads)
        if (sMe[i] < th && th <= sMe[i + 1]) s_bp = c0 + i;
      __syncthreads();
    }
    int bp = s_bp;
    if (bp < 0 && bk >= 0 && s_mek < th) bp = bk;  // the threshold inside the top-k bin
    ok = bp >= 0 && (bp == bk || (blo <= bp && bp <= bhi));
    if (ok) {
      unsigned long long in;
      const unsigned long long ktop = kk;
      auto pp = [&](unsigned long long K, int bin) { return bin == bp && (bp != bk || K >= ktop); };
      const unsigned long long mbp = bp == bk ? s_mek : me(bp);
      kcut = short_list ? rank_select(n, sKey, sBin, sF, pp, true, th - mbp, &in)
                        : radix_select(n, get, pp, true, th - mbp, M, a, S, &in);
      kept = mbp + in;
    }
  }
  if (a.min_p > 0.f) {  // a cut on the logit alone, after top-p
    const unsigned long long kmin = (unsigned long long)(~kinv) << 32;
    if (kmin > kcut) {
      kcut = kmin;
      kept = zmin;
    }
  }
  __syncthreads();
  // Consumed: the list, the prefix sums and the statistics words (every
  // call leaves them zero; past its capacity only kWideCandCap list entries
  // were written).
  for (int i = tid; i < (int)min(ncand, (unsigned)kWideCandCap); i += kThreads)
    const_cast<unsigned*>(cand)[i] = 0;
  if (bins)
    for (int i = tid; i < kWideBins; i += kThreads) {
      gh[i] = 0;
      if (count_cut) gc[i] = 0;
    }
  for (int u = tid; u < a.nsplit; u += kThreads) a.ws.stats[(size_t)rr * a.nsplit + u] = 0;
  if (tid == 0) {
    if (!ok) {  // the selection's bins disagree (not expected): the request fails closed
      set_status(a.ws.status, SPEC_ELIMIT);
      atomicExch(&a.ws.sync[b].failed, 1);
    }
    wr->kcut = kcut;
    wr->Z = (float)((double)kept * 0x1p-40);
    wr->zmin = 0;
    wr->kmin_inv = 0;
    wr->ncand = 0;
  }
}

// ------------------------------------------------------------------ 6
template <int DT, bool VEC>
__device__ __forceinline__ void wide_draw_item(const ChainArgs& a, int b, int part) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  __shared__ float sP[SPEC_MAX_DRAFT], sQ[SPEC_MAX_DRAFT], sU[SPEC_MAX_DRAFT + 1];
  __shared__ int sJ, sBad, sLast, sFailed;
  __shared__ unsigned long long sWT[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = a.k;
  const size_t row_bytes = (size_t)a.V * ES;
  const WideRow* rec = a.ws.wrow + (size_t)b * a.rows;  // target rows 0..k, then draft rows

  const int kraw = a.draft_lens ? a.draft_lens[b] : k;
  const bool bad_len = kraw < 0 || kraw > k;
  const int kb = bad_len ? 0 : kraw;
  if (tid == 0) sBad = bad_len;
  if (tid <= k)
    sU[tid] = a.uniforms ? a.uniforms[(size_t)b * (k + 1) + tid]
                         : philox_uniform(a.seeds[b], a.offsets[b], tid);
  __syncthreads();
  if (tid < kb) {  // p'(x_i) and q'(x_i) on the filtered rows
    const int x = a.tokens[(size_t)b * k + tid];
    if (x < 0 || x >= a.V) {
      sBad = 1;
    } else {
      const float xp = load_logit<DT>(a.target + ((size_t)b * (k + 1) + tid) * row_bytes, x);
      const float xq = load_logit<DT>(a.draft + ((size_t)b * k + tid) * row_bytes, x);
      const WideRow rp = rec[tid], rq = rec[k + 1 + tid];
      sP[tid] = make_key(xp, x) >= rp.kcut ? ex2(scaled(xp - rp.M, a.c_hi, a.c_lo)) / rp.Z : 0.f;
      sQ[tid] = make_key(xq, x) >= rq.kcut ? ex2(scaled(xq - rq.M, a.c_hi, a.c_lo)) / rq.Z : 0.f;
    }
  }
  __syncthreads();
  if (warp == 0) {  // accept scan: r_i < p'_i / q'_i, q' == 0 accepts; j = first reject
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
  CutMask cut{0, 0};
  if (j >= 0) {
    const WideRow rp = rec[j];
    prow = a.target + ((size_t)b * (k + 1) + j) * row_bytes;
    mp = rp.M;
    cut.kp = rp.kcut;
    if (j < kb) {
      const WideRow rq = rec[k + 1 + j];
      qrow = a.draft + ((size_t)b * k + j) * row_bytes;
      mq = rq.M;
      cut.kq = rq.kcut;
      lam = rp.Z / rq.Z;  // max(0, p' - q') = max(0, e_p - lam e_q) / Z_p
    }
    const int c0 = part * a.cpc, c1 = min(a.nchunks, c0 + a.cpc);
    const unsigned long long wt = chunk_sums<DT, VEC, false, true>(
        a, prow, qrow, c0, c1, mp, mq, lam, a.ws.chunks + (size_t)b * a.nchunks, TokenMask{nullptr, 0}, cut);
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

  // Every item has read the request's row records: return them to zero.
  for (int i = tid; i < a.rows * (int)(sizeof(WideRow) / 4); i += kThreads)
    reinterpret_cast<unsigned*>(const_cast<WideRow*>(rec))[i] = 0;
  int32_t* out = a.out_tokens + (size_t)b * (k + 1);
  if (j < 0 || sFailed) {  // a bad draft token or length, or a failed cut: fail closed
    for (int i = tid; i < a.nchunks; i += kThreads) a.ws.chunks[(size_t)b * a.nchunks + i] = 0;
    for (int i = tid; i < a.nsplit2; i += kThreads) a.ws.items[(size_t)b * a.nsplit2 + i] = 0;
    for (int i = tid; i <= k; i += kThreads) out[i] = -1;
    if (a.out_probs)
      for (int i = tid; i < 2 * k; i += kThreads) a.out_probs[(size_t)b * 2 * k + i] = NAN;
    if (tid == 0) {
      a.out_n[b] = -1;
      set_status(a.ws.status, j < 0 ? SPEC_EBADINDEX : SPEC_ELIMIT);
    }
    return;
  }
  if (a.out_probs && tid < k) {  // padded positions are not verified: NaN
    a.out_probs[((size_t)b * k + tid) * 2] = tid < kb ? sP[tid] : NAN;
    a.out_probs[((size_t)b * k + tid) * 2 + 1] = tid < kb ? sQ[tid] : NAN;
  }
  const double u = (double)sU[kb];
  const int tok = draw_token<DT, VEC, false, true>(a, b, prow, qrow, mp, mq, lam, u, TokenMask{nullptr, 0}, cut);
  for (int i = tid; i <= k; i += kThreads)
    out[i] = i < j ? a.tokens[(size_t)b * k + i] : (i == j ? tok : -1);
  if (tid == 0) {
    a.out_n[b] = j;
    if (a.seq_lens) a.seq_lens[b] += j + 1;
  }
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) wide_draw_kernel(const ChainArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int items = a.B * a.nsplit2;
  for (int h = blockIdx.x; h < items; h += gridDim.x) {
    const int b = h / a.nsplit2;
    wide_draw_item<DT, VEC>(a, b, h - b * a.nsplit2);
    __syncthreads();
  }
}

template <class K>
cudaError_t launch_dep(K kernel, long grid, const ChainArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// The current device's SM count (cached per device).
cudaError_t sm_count(int* out) {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    e = cudaDeviceGetAttribute(&cached[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  *out = cached[dev];
  return cudaSuccess;
}

template <int DT, bool VEC>
cudaError_t wide_draw_grid(int* grid) {
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
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wide_draw_kernel<DT, VEC>, kThreads, 0);
    if (e != cudaSuccess) return e;
    cached[dev] = sms * (per_sm > 0 ? per_sm : 1);
  }
  *grid = cached[dev];
  return cudaSuccess;
}

template <int DT, bool VEC>
cudaError_t launch_wide_t(const ChainArgs& args, cudaStream_t st) {
  int slots = 0;
  cudaError_t e = wide_draw_grid<DT, VEC>(&slots);
  if (e != cudaSuccess) return e;
  ChainArgs a = args;
  while ((long)a.B * a.nsplit2 > slots && a.cpc < a.nchunks) {  // as the chain's draw
    a.cpc *= 2;
    a.nsplit2 = ceil_div(a.nchunks, a.cpc);
  }
  const long rows = (long)a.B * a.rows;
  const long slices = rows * a.nsplit;
  const long items = (long)a.B * a.nsplit2;
  if ((e = launch_first(chain_rowstats_kernel<DT, VEC>, slices, kThreads, st, a)) != cudaSuccess) return e;
  const bool cnt = a.top_k > 0, mp = a.min_p > 0.f;
  // Slices per histogram CTA: up to kHistSlices, while the grid still fills
  // every SM with four CTAs.
  int sms = 0;
  if ((e = sm_count(&sms)) != cudaSuccess) return e;
  const long spc = std::max(1L, std::min((long)kHistSlices, slices / (4L * sms)));
  const long hist = rows * ((a.nsplit + spc - 1) / spc);
  if (cnt)
    e = mp ? launch_dep(wide_hist_kernel<DT, VEC, true, true, true>, hist, a, st)
           : launch_dep(wide_hist_kernel<DT, VEC, true, false, true>, hist, a, st);
  else if (a.top_p < 1.f)
    e = mp ? launch_dep(wide_hist_kernel<DT, VEC, false, true, true>, hist, a, st)
           : launch_dep(wide_hist_kernel<DT, VEC, false, false, true>, hist, a, st);
  else  // min_p alone
    e = launch_dep(wide_hist_kernel<DT, VEC, false, true, false>, hist, a, st);
  if (e != cudaSuccess) return e;
  if (cnt || a.top_p < 1.f) {  // (min_p alone: no bins, no candidates)
    // one histogram CTA per row runs the bins step itself
    if (hist > rows) {
      e = cnt ? launch_dep(wide_bins_kernel<DT, VEC, true>, rows, a, st)
              : launch_dep(wide_bins_kernel<DT, VEC, false>, rows, a, st);
      if (e != cudaSuccess) return e;
    }
    if ((e = launch_dep(wide_cand_kernel<DT, VEC>, slices, a, st)) != cudaSuccess) return e;
  }
  if ((e = launch_dep(wide_cut_kernel<DT>, rows, a, st)) != cudaSuccess) return e;
  return launch_dep(wide_draw_kernel<DT, VEC>, items < slots ? items : slots, a, st);
}

}  // namespace

cudaError_t launch_wide(const ChainArgs& a, int dtype, bool vec, cudaStream_t st) {
  if (dtype == SPEC_BF16)
    return vec ? launch_wide_t<SPEC_BF16, true>(a, st) : launch_wide_t<SPEC_BF16, false>(a, st);
  return vec ? launch_wide_t<SPEC_F32, true>(a, st) : launch_wide_t<SPEC_F32, false>(a, st);
}

}  // namespace sv
