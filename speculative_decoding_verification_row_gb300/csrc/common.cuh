// Device helpers shared by the verification kernels (sm_103a).
//
// Work decomposition used by every logit-streaming kernel: a logit row of V
// elements is read as "vectors" (16 bytes = 8 bf16 or 4 fp32 when every row
// starts 16-byte aligned, else single elements) and cut into equal "units" of
// at most kThreads * kVecPerThread vectors (32 KB of bf16/fp32).  One CTA
// reads one unit with every thread issuing all of its (up to 8) 128-bit loads
// before using any, so 32 KB per CTA are in flight.  CTAs are numbered
// request-major, so the units of one request are dispatched together and
// the per-request epilogue (run by the request's last CTA, found with an
// atomic ticket; nothing ever waits) overlaps with other requests' streaming.
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
constexpr int kChunksPerCta = 32;   // chunks one sampling CTA sums (4 per warp)

struct ReqInfo {        // per-request result of the accept scan, read by the sampler
  int j;                // first rejected position, k = all accepted, -1 = failed
  int pad;
  float mp, sp;         // max and sum-exp of target row j
  float mq, sq;         // max and sum-exp of draft row j (residual only)
  float pad2[2];
};
static_assert(sizeof(ReqInfo) == 32, "ReqInfo layout");

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
__host__ __device__ inline int ceil_div(long a, long b) { return (int)((a + b - 1) / b); }
// Units per row for the worst case (one element per vector).
__host__ __device__ inline int max_splits(int V) { return ceil_div(V, kUnitVecs); }
__host__ __device__ inline int num_chunks(int V) { return ceil_div(V, kChunk); }

// Byte offsets of the workspace regions for one call's sizes.
struct WsLayout {
  size_t status, tick1, tick2, part, req, chunks, total;
  __host__ __device__ WsLayout(int B, int rows, int V) {
    size_t off = 0;
    status = off; off += 256;
    tick1 = off; off += align256(sizeof(int) * (size_t)B);
    tick2 = off; off += align256(sizeof(int) * (size_t)B);
    part = off; off += align256(sizeof(float2) * (size_t)B * rows * max_splits(V));
    req = off; off += align256(sizeof(ReqInfo) * (size_t)B);
    chunks = off; off += align256(sizeof(float) * (size_t)B * num_chunks(V));
    total = off;
  }
};

struct Ws {  // typed views of one call's workspace
  int* status;
  int* tick1;
  int* tick2;
  float2* part;
  ReqInfo* req;
  float* chunks;
};

inline Ws ws_views(void* base, const WsLayout& l) {
  char* p = static_cast<char*>(base);
  return Ws{reinterpret_cast<int*>(p + l.status), reinterpret_cast<int*>(p + l.tick1),
            reinterpret_cast<int*>(p + l.tick2), reinterpret_cast<float2*>(p + l.part),
            reinterpret_cast<ReqInfo*>(p + l.req), reinterpret_cast<float*>(p + l.chunks)};
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

// ---------------------------------------------------------------- (max, sum-exp) merge
// Merge two partial softmax statistics (m, s) with s = sum 2^(c (x - m)).
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2, float c_hi,
                                          float c_lo) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) {
    m = M;
    s = 0.f;
    return;
  }
  s = s * ex2(scaled(m - M, c_hi, c_lo)) + s2 * ex2(scaled(m2 - M, c_hi, c_lo));
  m = M;
}

// Record the first data-dependent error of a call.
__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// Ticket of the threadfence-reduction pattern: returns true in exactly one CTA
// of the `expected` CTAs that call it for the same counter (the last to
// arrive), which then resets the counter for the next call.  No CTA waits.
__device__ __forceinline__ bool last_arrival(int* counter, int expected) {
  __shared__ int s_last;
  __threadfence();  // this thread's global writes are visible device-wide
  __syncthreads();
  if (threadIdx.x == 0) {
    const int t = atomicAdd(counter, 1);
    s_last = (t == expected - 1);
    if (s_last) *counter = 0;
  }
  __syncthreads();
  if (s_last) __threadfence();  // order the epilogue's reads after the ticket
  return s_last != 0;
}

}  // namespace sv
