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

#include "draw.cuh"

namespace sv {

namespace {

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
  // Merge the slice statistics of every row of the request as they arrive:
  // thread r takes row r, issues the loads of its words (eight at a time)
  // before using any, waiting only for words still 0, then adds
  // S_s * 2^(c(m_s - M)) over its slices in slice order (one exp per slice).
  const unsigned long long* sb = a.ws.stats + (size_t)b * R * a.nsplit;
  bool to = false;  // a wait of this thread ran out
  for (int r = tid; r < rows; r += kThreads) {
    if (!used(r)) continue;
    const unsigned long long* pr = sb + (size_t)r * a.nsplit;
    float m = -INFINITY;
    for (int u0 = 0; u0 < a.nsplit; u0 += 8) {
      unsigned long long v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = u0 + q < a.nsplit ? ld_relaxed_u64(pr + u0 + q) : kNoStats;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
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
  if (k > 32) __syncthreads(); else __syncwarp();  // k <= 32: warp 0 wrote sP, sQ, sBad
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
  // One device-scope fence by thread 0 releases the whole CTA's sums before
  // the ticket: every chunk sum was written before the barrier above, which
  // made it visible to thread 0, and the fence is cumulative over them.
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
  const long g1 = (long)a.B * a.rows * a.nsplit;
  if (!skip_pass1) {
    e = launch_first(chain_rowstats_kernel<DT, VEC>, g1, kThreads, st, a);
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
