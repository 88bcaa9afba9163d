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
// those sums are exact whatever their order; the tail below the depth D0
// (step 2) is summed in fp32 per thread, at most (1 - top_p) Z / 2 in all, so
// its rounding stays far inside the oracle's 1e-6 near-tie window.  Six
// stream-ordered grids, each a programmatic dependent that waits for its
// predecessor before reading (no polling):
//   1. chain_rowstats_kernel (the chain's pass 1): the slice maxima and sums.
//   2. wide_hist_kernel, one CTA per 32 KB slice: each token's bin
//      floor(32 c (M - x)) (2048 bins of 1/32 of a log2 unit, the last
//      holding everything below) and mass, into a shared-memory histogram
//      (counts too when top-k cuts), then into the row's; the mass and the
//      smallest logit key of the tokens with e_t >= min_p.  Without a top-k
//      cut only tokens above a depth D0 get their own bin: the V tokens
//      below it weigh at most V 2^-D0 = (1 - top_p) Z / 2, so the top-p cut
//      cannot fall among them; their mass goes into the last bin (on the
//      headline shape D0 leaves ~13 % of the tokens heavy; each warp queues
//      its heavy tokens by ballot and adds them 32 at a time).  min_p alone
//      needs no bins.
//   3. wide_bins_kernel, one CTA per row: prefix sums over the bins give
//      the bin where the top-k count is reached and the range of bins the
//      top-p threshold can fall in (the top-k mass is known to within the
//      top-k bin); the bins are rewritten as their exclusive prefix sums.
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
// BINS = false (min_p alone): no histogram, only the min_p mass and key.
template <int DT, bool VEC, bool COUNT, bool MINP, bool BINS>
__global__ void __launch_bounds__(kThreads, 4) wide_hist_kernel(const ChainArgs a) {
  // The slice's bin masses in three 14-bit parts of the 2^-40 fixed point
  // (32-bit shared adds; a slice holds at most 2^14 tokens, so each part's
  // sum stays below 2^28), recombined exactly at the end.
  __shared__ unsigned hm[3][kWideBins];
  __shared__ unsigned hc[COUNT ? kWideBins : 1];
  __shared__ unsigned long long s_z[kWarps];
  __shared__ unsigned s_k[kWarps];
  using IO = Io<DT, VEC>;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rr = blockIdx.x / a.nsplit, s = blockIdx.x - rr * a.nsplit;
  int b, r;
  slice_row(a, rr, b, r);
  for (int i = tid; i < kWideBins; i += kThreads) {
    hm[0][i] = hm[1][i] = hm[2][i] = 0u;
    if (COUNT) hc[i] = 0;
  }
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
    if (v < vend) {
      IO::load(row, v, w[u]);
    } else {  // past the row: -inf (no mass; not counted, see below)
#pragma unroll
      for (int q = 0; q < IO::NW; ++q) w[u][q] = (VEC && DT == SPEC_BF16) ? 0xff80ff80u : 0xff800000u;
    }
  }
  float Zs;
  const float M = row_stats(a, rr, &Zs);  // also orders the clearing above before the adds
  const float cR = a.c_rn * (float)kWideBinsPerLog2;
  // Bins from b0 on take the light tokens, summed in registers (no top-k
  // cut: the top-p cut lies above depth D0; min_p alone needs no bins).
  int b0 = kWideBins;
  if (!COUNT) {
    if (a.top_p < 1.f) {
      const float D0 = log2f((float)a.V / ((1.f - a.top_p) * fmaxf(Zs, 1.f))) + 1.f;
      const float fb = ceilf(D0 * (float)kWideBinsPerLog2) + 1.f;
      b0 = fb < 1.f ? 1 : (fb >= (float)(kWideBins - 1) ? kWideBins - 1 : (int)fb);
    } else {
      b0 = 0;
    }
  }
  if (s == 0 && tid == 0) {  // every slice of the row computes the same
    a.ws.wrow[rr].b0 = b0;
    a.ws.wrow[rr].M = M;
  }
  const float fb0 = (float)b0;
  unsigned long long zmin = 0;
  unsigned kinv = 0;
  float light = 0.f;  // light tokens' mass: each < 2^-D0, summed in fp32 per thread
  // Heavy tokens of each vector (8 or 4 per lane) are packed per warp by
  // ballot into a shared queue as (bin, mass) and added to the histogram
  // after the vector, one per lane: a warp-wide 64-bit shared add costs
  // about the same however few of its lanes are active, so one add per 32
  // heavy tokens instead of one per token position.
  // (with a top-k count cut every token is heavy: no queue, direct adds)
  __shared__ unsigned qbin[COUNT ? 1 : kWarps][COUNT ? 1 : 32 * IO::EPV];
  __shared__ float qe[COUNT ? 1 : kWarps][COUNT ? 1 : 32 * IO::EPV];
  auto add_mass = [&](unsigned bin, float e) {
    const unsigned long long f = to_fixed(e * 256.f);  // < 2^41
    if (f) {
      atomicAdd(&hm[0][bin], (unsigned)f & 0x3fffu);
      atomicAdd(&hm[1][bin], (unsigned)(f >> 14) & 0x3fffu);
      atomicAdd(&hm[2][bin], (unsigned)(f >> 28));
    }
  };
  const unsigned below = (1u << lane) - 1u;
  const float2 nM = make_float2(-M, -M), chi = make_float2(a.c_hi, a.c_hi), clo = make_float2(a.c_lo, a.c_lo),
               ncR = make_float2(-cR, -cR);
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    float x[IO::EPV];
    IO::unpack(w[u], x);
    int qn = 0;  // warp-uniform
#pragma unroll
    for (int i = 0; i < IO::EPV; i += 2) {
      // two tokens at a time in packed fp32x2: d = x - M, the exponent
      // scaled(d) = d c_hi + d c_lo and the bin (M - x) cR = d (-cR), each
      // the same rounding as the scalar operations of mass_fix / mass_bin
      const float x1 = i + 1 < IO::EPV ? x[i + 1 < IO::EPV ? i + 1 : i] : -INFINITY;  // (EPV may be 1)
      const float2 d = add2(make_float2(x[i], x1), nM);
      const float2 y = fma2(d, chi, mul2(d, clo));
      const float2 fb = mul2(d, ncR);
      const float e2[2] = {ex2(y.x), ex2(y.y)};
      const float fbin2[2] = {fb.x, fb.y};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (i + h >= IO::EPV) break;
        const float e = e2[h], fbin = fbin2[h];
        if constexpr (MINP) {
          if (e >= a.min_p) {
            zmin += to_fixed(e * 256.f);
            kinv = max(kinv, ~ord32(h ? x1 : x[i]));
          }
        }
        if constexpr (!BINS) {
          // min_p alone: the cut is the smallest key with e >= min_p
        } else if constexpr (COUNT) {  // every token of the row is counted
          if (vbeg + tid + u * kThreads < vend) {
            const unsigned bin = (unsigned)(int)fminf(fbin, (float)(kWideBins - 1));
            add_mass(bin, e);
            atomicAdd(&hc[bin], 1u);
          }
        } else {  // past the row: x = -inf, so fbin = +inf, light, no mass
          const bool heavy = fbin < fb0;
          light += heavy ? 0.f : e;
          const unsigned hmask = __ballot_sync(0xffffffffu, heavy);
          if (heavy) {
            const int slot = qn + __popc(hmask & below);
            qbin[warp][slot] = __float_as_uint(fbin);
            qe[warp][slot] = e;
          }
          qn += __popc(hmask);
        }
      }
    }
    if constexpr (!COUNT && BINS) {
      __syncwarp();
      for (int q = lane; q < qn; q += 32)
        add_mass((unsigned)(int)__uint_as_float(qbin[warp][q]), qe[warp][q]);  // fbin < b0 <= 2047
      __syncwarp();
    }
  }
  unsigned long long* gh = a.ws.whist + (size_t)rr * kWideBins;
  unsigned* gc = a.ws.wcount + (size_t)rr * kWideBins;
  if (b0 < kWideBins) {  // the light tokens' mass, into the last bin
    unsigned long long tot;
    block_excl_u64(to_fixed(light * 256.f), &tot);  // (its barriers also order the adds above)
    if (tid == 0 && tot) atomicAdd(gh + kWideBins - 1, tot);
  } else {
    __syncthreads();
  }
  for (int i = tid; i < min(b0, kWideBins); i += kThreads) {
    const unsigned long long m = ((unsigned long long)hm[2][i] << 28) + ((unsigned long long)hm[1][i] << 14) + hm[0][i];
    if (m) atomicAdd(gh + i, m);
    if (COUNT && hc[i]) atomicAdd(gc + i, hc[i]);
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
      WideRow* wr = a.ws.wrow + rr;
      if (z) atomicAdd(&wr->zmin, z);
      if (kk) atomicMax(&wr->kmin_inv, kk);
    }
  }
}

// ------------------------------------------------------------------ 3
// Bins b of a row are held 8 per thread (thread t: 8t .. 8t + 7).
constexpr int kBinsPerThread = kWideBins / kThreads;
static_assert(kBinsPerThread * kThreads == kWideBins, "bins per thread");

__global__ void __launch_bounds__(kThreads) wide_bins_kernel(const ChainArgs a) {
  __shared__ int s_bk, s_blo, s_bhi;
  __shared__ unsigned long long s_mb, s_mbin;
  const int tid = threadIdx.x;
  const int rr = blockIdx.x, b = rr / a.rows, r = rr - b * a.rows;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (a.draft_lens && !row_used(a.k, a.draft_lens[b], r)) return;
  unsigned long long* gh = a.ws.whist + (size_t)rr * kWideBins + kBinsPerThread * tid;
  unsigned* gc = a.ws.wcount + (size_t)rr * kWideBins + kBinsPerThread * tid;
  const bool count_cut = a.top_k > 0;
  unsigned long long m[kBinsPerThread], tm = 0, tc = 0;
  unsigned c[kBinsPerThread];
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    m[j] = gh[j];
    c[j] = count_cut ? gc[j] : 0u;
    tm += m[j];
    tc += c[j];
  }
  if (tid == 0) {
    s_bk = s_blo = s_bhi = -1;
    s_mb = 0;
    s_mbin = 0;
  }
  unsigned long long Z, N;
  const unsigned long long pm = block_excl_u64(tm, &Z);
  const unsigned long long pc = block_excl_u64(tc, &N);
  // top-k: the bin where the running count reaches top_k
  if (count_cut && (unsigned long long)a.top_k < N) {
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
      if (count_cut) gc[j] = (unsigned)cb;
      mb += m[j];
      cb += c[j];
    }
  }
  __syncthreads();
  if (tid == 0) {
    WideRow* wr = a.ws.wrow + rr;
    wr->bk = s_bk;
    wr->blo = s_blo;
    wr->bhi = s_blo >= 0 ? s_bhi : -1;
    wr->ztot = Z;
  }
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
  const int bk = wr->bk, blo = wr->blo, bhi = wr->bhi, b0 = wr->b0;
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
  if (cnt)
    e = mp ? launch_dep(wide_hist_kernel<DT, VEC, true, true, true>, slices, a, st)
           : launch_dep(wide_hist_kernel<DT, VEC, true, false, true>, slices, a, st);
  else if (a.top_p < 1.f)
    e = mp ? launch_dep(wide_hist_kernel<DT, VEC, false, true, true>, slices, a, st)
           : launch_dep(wide_hist_kernel<DT, VEC, false, false, true>, slices, a, st);
  else  // min_p alone
    e = launch_dep(wide_hist_kernel<DT, VEC, false, true, false>, slices, a, st);
  if (e != cudaSuccess) return e;
  if ((e = launch_dep(wide_bins_kernel, rows, a, st)) != cudaSuccess) return e;
  if ((e = launch_dep(wide_cand_kernel<DT, VEC>, slices, a, st)) != cudaSuccess) return e;
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
