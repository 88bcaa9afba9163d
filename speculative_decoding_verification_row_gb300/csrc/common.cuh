// Device helpers shared by the verification kernels (sm_103a).
//
// Work decomposition used by every logit-streaming kernel: a logit row of V
// elements is read as "vectors" (16 bytes = 8 bf16 or 4 fp32 when every row
// starts 16-byte aligned, else single elements) and cut into equal "units" of
// at most kThreads * kVecPerThread vectors (32 KB of bf16/fp32).  One CTA
// reads one unit with every thread issuing all of its (up to 8) 128-bit loads
// before using any, so 32 KB per CTA are in flight.  CTAs are numbered
// request-major, so the units of one request are dispatched together.  A
// streaming CTA publishes its unit's result as one nonzero 64-bit word and
// exits (no fence, no counter); a second grid, launched as a programmatic
// dependent, polls each request's words and finishes the request.
#pragma once

#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

constexpr int kThreads = 256;       // threads per CTA of every streaming kernel
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 8;    // vectors a thread holds in registers
constexpr int kUnitVecs = kThreads * kVecPerThread;
constexpr int kChunk = 256;         // elements per inverse-CDF chunk (32 lanes x 8)
constexpr int kChunksPerCta = 64;   // chunks of one draw item, at least (the launch may double it)


__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
__host__ __device__ inline int ceil_div(long a, long b) { return (int)((a + b - 1) / b); }
// Units per row for the worst case (one element per vector).
__host__ __device__ inline int max_splits(int V) { return ceil_div(V, kUnitVecs); }
__host__ __device__ inline int num_chunks(int V) { return ceil_div(V, kChunk); }
__host__ __device__ inline int num_items(int V) { return ceil_div(num_chunks(V), kChunksPerCta); }

// Per-request synchronisation words, 64 bytes apart so that the CTAs of
// different requests rarely share a line.
struct ReqSync {
  int tick2;   // chain: draw items (filtered: row CTAs) of the request that have finished
  int failed;  // nonzero once a wait of the request's second phase ran out
  int pad[14];
};
static_assert(sizeof(ReqSync) == 64, "ReqSync layout");

__host__ __device__ inline size_t stats_bytes(int B, int rows, int V) {
  return sizeof(unsigned long long) * (size_t)B * rows * max_splits(V);
}

// Byte offsets of the workspace regions for one call's sizes.  The status
// word and the sync lines of SPEC_MAX_BATCH requests come first, at offsets
// that do not depend on the call.  The regions after them move with the
// call's sizes, so one call's scratch may sit where another call's slice
// statistics sit; hence every call returns everything it writes (sync lines,
// statistics, partials, sums) to zero before it ends, and the whole
// workspace but the status word is zero between calls.  The chain path's
// statistics words rely on it: an entry is zero until its slice writes it
// (a written entry never is: see stats_pack).
struct WsLayout {
  size_t status, sync, stats, part, chunks, items, total;
  __host__ __device__ WsLayout(int B, int rows, int V) {
    size_t off = 0;
    status = off; off += 256;
    sync = off; off += sizeof(ReqSync) * (size_t)SPEC_MAX_BATCH;
    stats = off; off += align256(stats_bytes(B, rows, V));
    part = off; off += align256(sizeof(float2) * (size_t)B * rows * max_splits(V));
    chunks = off; off += align256(sizeof(unsigned long long) * (size_t)B * num_chunks(V));
    items = off; off += align256(sizeof(unsigned long long) * (size_t)B * num_items(V));
    total = off;
  }
};

// Exact filtering of any kept-set size (top-p or min_p without top-k, top-k
// above SPEC_MAX_TOPK): each row's mass histogram over kWideBins bins of
// 1/kWideBinsPerLog2 of a log2 unit below the row maximum (the last bin
// holds the rest; once the bins are chosen it holds exclusive prefix sums),
// its candidate list (the tokens of the bins a cut can fall in) and its
// record.
constexpr int kWideBinsPerLog2 = 32;
constexpr int kWideBins = 2048;
constexpr int kWideCandCap = 4096;  // candidates listed per row; a row with more rescans itself
struct WideRow {
  unsigned long long zmin;  // sum of the fixed-point masses with 2^(c(x - M)) >= min_p
  unsigned kmin_inv;        // ~ the smallest order key (ord32) among those tokens
  unsigned ncand;           // tokens appended to the row's candidate list
  int bk, blo, bhi;         // the top-k bin, the top-p bin range (-1: none)
  int b0;                   // bins >= b0 are merged into the last bin (light tokens)
  unsigned long long kcut;  // token t is kept iff make_key(x_t, t) >= kcut
  float M, Z;               // row maximum and (after the cut) kept mass, 2^(c(x - M)) units
  unsigned long long ztot;  // the row's total fixed-point mass
  int pad1[2];
};
static_assert(sizeof(WideRow) == 64, "WideRow layout");

struct Ws {  // typed views of one call's workspace
  int* status;                 // first word of the 256-byte status block
  ReqSync* sync;
  unsigned long long* stats;   // chain: packed (M, S) of each row slice, 0 = not yet written
  float2* part;                // argmax: each unit's packed (max, index + 1)
  unsigned long long* chunks;  // draw-weight sum of each 256-token chunk, in 2^-32 units
  unsigned long long* items;   // sum of each draw item's chunks, in 2^-32 units
  unsigned long long* cand;    // filtered: each row's kept list
  float* pq;                   // filtered: p_i(x_i) and q_i(x_i) of each request
  unsigned short* codes;       // filtered: each slice thread's largest-logit prefix
  unsigned long long* whist;   // wide filter: per row kWideBins fixed-point masses (2^-40)
  unsigned* wcount;            // wide filter: per row kWideBins token counts (top-k cut)
  WideRow* wrow;               // wide filter: per row record
  unsigned* wcand;             // wide filter: per row kWideCandCap candidate token ids
};

// The filtered chain path appends three regions to the chain layout: per
// row, its kept list (top_k words); per request 2k draft-token
// probabilities; per slice thread (worst case of max_splits(V) slices per
// row), the 16-bit prefix of its largest logit.
struct FilterLayout {
  size_t cand, pq, codes, total;
  __host__ __device__ FilterLayout(int B, int k, int V, int top_k) {
    size_t off = WsLayout(B, 2 * k + 1, V).total;
    cand = off; off += align256(sizeof(unsigned long long) * (size_t)B * (2 * k + 1) * top_k);
    pq = off; off += align256(sizeof(float) * (size_t)B * 2 * k);
    codes = off; off += align256(sizeof(unsigned short) * (size_t)B * (2 * k + 1) * max_splits(V) * kThreads);
    total = off;
  }
};

// The wide filtered path appends its per-row regions to the chain layout.
struct WideLayout {
  size_t hist, count, rec, cand, total;
  __host__ __device__ WideLayout(int B, int k, int V) {
    const size_t rows = (size_t)B * (2 * k + 1);
    size_t off = WsLayout(B, 2 * k + 1, V).total;
    hist = off; off += align256(sizeof(unsigned long long) * rows * kWideBins);
    count = off; off += align256(sizeof(unsigned) * rows * kWideBins);
    rec = off; off += align256(sizeof(WideRow) * rows);
    cand = off; off += align256(sizeof(unsigned) * rows * kWideCandCap);
    total = off;
  }
};

inline Ws ws_views(void* base, const WsLayout& l) {
  char* p = static_cast<char*>(base);
  return Ws{reinterpret_cast<int*>(p + l.status), reinterpret_cast<ReqSync*>(p + l.sync),
            reinterpret_cast<unsigned long long*>(p + l.stats),
            reinterpret_cast<float2*>(p + l.part),
            reinterpret_cast<unsigned long long*>(p + l.chunks),
            reinterpret_cast<unsigned long long*>(p + l.items), nullptr, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr};
}

// ---------------------------------------------------------------- loads
// Streaming loads: read-only path, not kept in L1.
__device__ __forceinline__ void ld_stream_v4(const void* p, uint32_t (&w)[4]) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 2^x on the SFU (MUFU.EX2).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(e)/T * d, with log2(e)/T carried as c_hi + c_lo (c_hi rounded down,
// 0 < c_lo): the constant's rounding then costs no systematic error, and
// d = -inf still gives -inf.
__device__ __forceinline__ float scaled(float d, float c_hi, float c_lo) {
  return fmaf(d, c_hi, d * c_lo);
}

// -m * c rounded to fp32 for the one-fma exponent 2^(x c + o): returns o
// and, in *eps, its rounding error (-m c - o, exact by the product's fma),
// so that 2^(x c - m c) = 2^(x c + o) * 2^(-eps) up to the exponent's final
// rounding.  m = -inf is not passed (callers use 0 for an empty set).
__device__ __forceinline__ float fma_offset(float m, float c, float* eps) {
  const float o = -m * c;
  *eps = fmaf(-m, c, -o);
  return o;
}

// Order keys: ord32 is monotone in the logit (-0 and +0 alike);
// make_key(x, t) orders tokens by (logit descending, token ascending) as
// decreasing 64-bit keys.
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

// One stored logit widened to fp32 (exact for both dtypes).
template <int DT>
__device__ __forceinline__ float load_logit(const char* row, long t) {
  if (DT == SPEC_BF16)
    return __uint_as_float(uint32_t(reinterpret_cast<const unsigned short*>(row)[t]) << 16);
  return reinterpret_cast<const float*>(row)[t];
}

// Vector I/O of one dtype: VEC = 16-byte vectors, else one element per vector.
template <int DT, bool VEC>
struct Io {
  static constexpr int ES = DT == SPEC_BF16 ? 2 : 4;          // element bytes
  static constexpr int EPV = VEC ? 16 / ES : 1;               // elements per vector
  static constexpr int NW = VEC ? 4 : 1;                      // 32-bit words per vector

  __device__ __forceinline__ static void load(const char* row, long v, uint32_t (&w)[NW]) {
    if constexpr (VEC) {
      ld_stream_v4(row + v * 16, w);
    } else if constexpr (DT == SPEC_BF16) {
      w[0] = ld_stream_u16(row + v * 2) << 16;  // scalar bf16 kept in the high half
    } else {
      w[0] = ld_stream_u32(row + v * 4);
    }
  }

  __device__ __forceinline__ static void unpack(const uint32_t (&w)[NW], float (&e)[EPV]) {
    if constexpr (VEC && DT == SPEC_BF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        e[2 * i] = bf16_lo(w[i]);
        e[2 * i + 1] = bf16_hi(w[i]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < EPV; ++i) e[i] = __uint_as_float(w[i]);
    }
  }

  // Largest element of one vector.
  __device__ __forceinline__ static float vmax(const uint32_t (&w)[NW]) {
    if constexpr (VEC && DT == SPEC_BF16) {
      uint32_t m = bf16x2_max(bf16x2_max(w[0], w[1]), bf16x2_max(w[2], w[3]));
      return fmaxf(bf16_lo(m), bf16_hi(m));
    } else {
      float e[EPV];
      unpack(w, e);
      float m = e[0];
#pragma unroll
      for (int i = 1; i < EPV; ++i) m = fmaxf(m, e[i]);
      return m;
    }
  }
};

// ---------------------------------------------------------------- packed fp32 pairs
// Blackwell executes add/mul/fma on fp32 pairs as one instruction.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " add.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(r.x), "=f"(r.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 r;
  asm("{\n .reg .b64 a, b, c, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %5};\n"
      " mov.b64 c, {%6, %7};\n fma.rn.f32x2 d, a, b, c;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return r;
}

// A non-negative weight sum (below 2^32) as an integer number of 2^-32,
// rounded to nearest even, with 32-bit conversions only (64-bit ones run on
// the FP64 pipe, which is narrow on this GPU).  x = h + f with h = trunc(x)
// and f = x - h exact; f * 2^32 < 2^32 - 255 is exact too, so rounding it
// rounds x * 2^32, and the tie parity is that of the low word.
__device__ __forceinline__ unsigned long long to_fixed(float x) {
  const unsigned h = __float2uint_rz(x);
  const unsigned l = __float2uint_rn((x - (float)h) * 4294967296.0f);
  return ((unsigned long long)h << 32) + l;
}

// ---------------------------------------------------------------- Philox
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11): ten rounds; a round takes the 64-bit products
// c0 * 0xD2511F53 and c2 * 0xCD9E8D57 and forms (hi2 ^ c1 ^ k0, lo2,
// hi0 ^ c3 ^ k1, lo0); the key advances by (0x9E3779B9, 0xBB67AE85) between
// rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo2 = 0xCD9E8D57u * c.z, hi2 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi2 ^ c.y ^ k0, lo2, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// Uniform i of a request's Philox stream: key = seed, counter = (offset,
// i / 4, 0); word i % 4, top 24 bits, scaled to [0, 1).
__device__ __forceinline__ float philox_uniform(unsigned long long seed, unsigned long long offset,
                                                int i) {
  const uint4 r = philox4x32_10(make_uint4((uint32_t)offset, (uint32_t)(offset >> 32),
                                           (uint32_t)(i / 4), 0u),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  const int w = i % 4;
  const uint32_t x = w == 0 ? r.x : w == 1 ? r.y : w == 2 ? r.z : r.w;
  return (float)(x >> 8) * (1.0f / 16777216.0f);
}

// Default upper bound of every device-side wait (about one second at 2 GHz).
// A wait that runs out sets SPEC_ETIMEOUT instead of spinning forever, and
// the request whose result depended on it fails closed.
constexpr long long kWaitCycles = 2000000000LL;

// Device-scope relaxed 64-bit accesses (single-copy atomic, no fence).
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
// Record the first data-dependent error of a call.
__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// Poll a word until a producer grid has written it (written words are never
// 0).  The producer was scheduled in full before the polling grid, so the
// wait ends; the bound (`limit` cycles) only turns a broken invariant into
// SPEC_ETIMEOUT, *timed_out = true and `on_timeout` instead of a hang.
static __device__ __noinline__ unsigned long long wait_word(const unsigned long long* p, int* status,
                                                            unsigned long long on_timeout,
                                                            long long limit, bool* timed_out) {
  unsigned long long v = ld_relaxed_u64(p);
  const long long t0 = clock64();
  while (!v) {
    if (clock64() - t0 > limit) {
      set_status(status, SPEC_ETIMEOUT);
      *timed_out = true;
      return on_timeout;
    }
    __nanosleep(64);
    v = ld_relaxed_u64(p);
  }
  return v;
}

}  // namespace sv
