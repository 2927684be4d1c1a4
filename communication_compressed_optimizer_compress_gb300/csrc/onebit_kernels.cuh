// onebit_kernels.cuh -- sm_103a kernels of the 1-bit Adam optimizer step.
//
// Method: "1-bit Adam: Communication Efficient Large-Scale Training with Adam's Convergence Speed"
// (Tang et al.), Sec. 4.3 (1-bit sign + magnitude-preserving scale), Sec. 6 and Sec. 11 (workers
// compress their momentum with error compensation, the server averages the messages and compresses
// again, the result is broadcast), and the AIMech page "1-bit Adam (Two-Stage Preconditioner-Frozen
// Error-Compensated Adam)" (v_t, m_t, V = diag(sqrt(v_Tw) + eps), x_t = x_{t-1} - gamma V^-1 m_hat).
//
// Data layout in HBM (one GPU simulates the n workers):
//   every per-element state array uses a padded layout in which tensor k starts at element
//   off_k = sum_{k'<k} roundup(L_k', 32); Dp = padded total, Wp = Dp / 32 sign words; worker sign
//   rows are Wr = roundup(Wp, 4) words apart, so every row starts on a 16-byte boundary.
//   m[Dp]        fp32 momentum (dense form: warm-up and the first compression step)
//   v[Dp]        fp32 variance; after the freeze den = sqrt(v) + eps
//   c[n][Dp]     fp32 compensated momentum c_i of the last step.  The worker error of that step is
//                delta_i = c_i - s_i*sign(c_i), recomputed from c_i and the last scale s_i with the
//                same single fp32 operation wherever it is needed, so it is never stored.
//   a[Dp]        fp32 server input of the last step; server error eps = a - S*sign(a), likewise.
//   wbits[n][Wr] worker sign words; sbits[Wp] server sign words (= the broadcast momentum's signs:
//                after a compression step m = S*sign(a) is represented by sbits and S, 1/8 B/elem).
//   scales       double-buffered by step parity: a step reads the previous step's scales (to rebuild
//                the errors and m) and writes its own.
//
// Work decomposition: host-built tables of chunks (<= kChunk elements, never crossing a tensor,
// starting on a 32-element boundary).  The server-side table never crosses a server shard either;
// the worker-side table is the same except inside tensors whose shards are shorter than a chunk,
// where one worker chunk holds several whole shards.  Each lane owns 8 consecutive elements
// (one byte of sign bits, one 256-bit load of fp32 state), so sign packing needs no cross-lane
// exchange and every warp access is a contiguous 1 KB (fp32) or 512 B (16-bit) span.
//
// Arithmetic: fp32 with explicit round-to-nearest intrinsics (no contraction into FMA), in the
// operation order of the method's formulas, so that the sign decisions match a plain CPU evaluation
// bit for bit.  Sums of squares are exact per element (double-float accumulation, promoted to fp64
// once per unit); the per-chunk partials are reduced in a fixed order (deterministic, independent
// of the grid size).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace onebit {

constexpr int kThreads = 256;          // threads per CTA of the streaming kernels
constexpr int kChunk = 65536;          // maximum elements per work chunk (multiple of 256)
constexpr int kMaxWorkers = 256;
constexpr int kScaleThreads = 256;     // threads per CTA of the scale kernels
constexpr int kWorkerUnroll = 3;       // 8-element groups whose loads a worker-kernel thread issues together

struct Chunk {
  int64_t off;    // element offset in the padded state layout (multiple of 32)
  int64_t uoff;   // element offset in the unpadded concatenation of the tensors
  int64_t start;  // element offset inside tensor `seg` (multiple of 32)
  int32_t seg;    // tensor k
  int32_t shard;  // server shard j of tensor k
  int32_t len;    // elements, 1..kChunk
  int32_t per;    // worker chunks only: the tensor's shard length S_k when the chunk spans several
                  // server shards (its groups then look up their own shard), else 0
};

struct Range {    // a contiguous run of chunks with its element count
  int32_t first;
  int32_t count;
  int64_t len;
};

struct StepArgs {
  const Chunk* chunks;       // server-side chunks: never cross a tensor or a server shard
  int32_t n_chunks;
  int32_t n;      // workers
  int32_t T;      // tensors
  int32_t pow2;   // n is a power of two: x / n == x * (1/n) exactly
  int64_t Dp;     // padded elements per row
  int64_t Wp;     // sign words per row
  int64_t Wr;     // worker sign-row stride in words (multiple of 4)
  const void* const* gptr;  // [n*T] gradient pointers, [worker][tensor]
  float* const* pptr;       // [T] parameter pointers
  float* m;
  float* v;
  float* c;
  float* a;
  uint32_t* wbits;
  uint32_t* sbits;
  const float* wscale_prev;  // [n*T]
  float* wscale_cur;         // [n*T]
  const float* sscale_prev;  // [T*n]
  float* sscale_cur;         // [T*n]
  double* wpart;             // [n*n_wchunks]
  double* spart;             // [n_chunks]
  const Range* seg_ranges;   // [T]   chunks of each tensor
  const Range* shard_ranges; // [T*n] chunks of each server shard
  unsigned int* status;
  float b1, omb1, b2, omb2, lr, eps, inv_n, nf, bc1, bc2;
  uint32_t stall_tx;  // test hook: extra bytes the staged kernels' copy barriers wait for (normally 0)
  const Chunk* wchunks;      // worker-side chunks: never cross a tensor; may span several shards
  const Range* wseg_ranges;  // [T]   worker chunks of each tensor
  int32_t n_wchunks;
  int32_t contig;            // the server kernel walks contiguous runs of chunks (many short segments)
  int64_t D;                 // elements (unpadded)
  int32_t nl;                // workers whose momentum this launch compresses (all n, or one rank's share)
  int32_t w0;                // the first of them: global workers w0 .. w0+nl-1 (c, wpart and gptr rows 0..nl-1)
#ifdef ONEBIT_CHECKS
  int64_t check_margin;      // test hook: padded elements the checks withhold from the end of the rows
#endif
};

// ------------------------------------------------------------------------------------------------
// Checked builds (compiled with -DONEBIT_CHECKS).  Before a kernel touches a unit of work (a chunk,
// a scale, an exchange range) it checks that the unit's descriptor keeps every access of the unit
// inside its buffers: the padded state rows in whole 32-element words (as the bulk copies read them),
// the caller's tensors, the sign rows, and the tensor, shard, worker and partial tables.  A unit that
// fails is skipped -- all threads of the block or warp that share it skip it together -- and the
// status word records it: bit 2, and bit 8 + the kernel's number (onebit_kernel_t).  Nothing traps.
// In normal builds the checks expand to nothing.

constexpr unsigned int kStatusBounds = 4u;

#ifdef ONEBIT_CHECKS
static __device__ __noinline__ void bounds_fail(unsigned int* status, int kernel) {
  atomicOr(status, kStatusBounds | (1u << (8 + kernel)));
}
// a chunk of the state: whole words inside the padded rows (less the test hook's margin), a valid
// tensor and shard, and its elements inside that tensor's caller buffers
__device__ __forceinline__ bool chunk_ok(const StepArgs& A, const Chunk& ch) {
  return ch.len > 0 && ch.len <= kChunk && ch.off >= 0 && (ch.off & 31) == 0 &&
         ch.off + ((ch.len + 31) & ~31) <= A.Dp - A.check_margin && ch.seg >= 0 && ch.seg < A.T &&
         ch.shard >= 0 && ch.shard < A.n && ch.start >= 0 && ch.start + ch.len <= A.wseg_ranges[ch.seg].len;
}
// a worker unit: its chunk, the shards its groups look up, and its worker row
__device__ __forceinline__ bool worker_unit_ok(const StepArgs& A, const Chunk& ch, int il) {
  return chunk_ok(A, ch) && ch.per >= 0 && (ch.per == 0 || ch.shard + (ch.len - 1) / ch.per < A.n) && il >= 0 &&
         il < A.nl && A.w0 >= 0 && A.w0 + il < A.n;
}
// a run of partials inside a table of `parts`
__device__ __forceinline__ bool range_ok(const Range& r, int64_t parts) {
  return r.first >= 0 && r.count >= 0 && (int64_t)r.first + r.count <= parts && r.len >= 0;
}
// inside a loop over units: skip this one
#define ONEBIT_CHECK_UNIT(ok, status, kernel) \
  if (!(ok)) {                                \
    ::onebit::bounds_fail(status, kernel);    \
    continue;                                 \
  }
// one item per thread group: give it up
#define ONEBIT_CHECK_ITEM(ok, status, kernel) \
  if (!(ok)) {                                \
    ::onebit::bounds_fail(status, kernel);    \
    return;                                   \
  }
// the staged kernels' chunk cursors: every role of the block moves its cursor past the same failing
// chunks (u, u + step, ... below end), so that the roles stay in step
__device__ __forceinline__ int skip_bad_chunks(const StepArgs& A, int u, int end, int step, int kernel) {
  for (; u < end && !chunk_ok(A, A.chunks[u]); u += step)
    if (threadIdx.x == 0) bounds_fail(A.status, kernel);
  return u;
}
#define ONEBIT_SKIP_BAD_CHUNKS(u, end, step, kernel) u = ::onebit::skip_bad_chunks(A, u, end, step, kernel)
#else
#define ONEBIT_CHECK_UNIT(ok, status, kernel)
#define ONEBIT_CHECK_ITEM(ok, status, kernel)
#define ONEBIT_SKIP_BAD_CHUNKS(u, end, step, kernel)
#endif

// ------------------------------------------------------------------------------------------------
// memory helpers (inline PTX): 256-bit accesses for fp32 state, 128-bit for 16-bit gradients.

__device__ __forceinline__ void ld8_stream(const float* p, float (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
               : "l"(p));
}
// coherent load for state the same kernel later overwrites in place
__device__ __forceinline__ void ld8_state(const float* p, float (&r)[8]) {
  asm volatile("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st8(float* p, const float (&r)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(r[0]), "f"(r[1]), "f"(r[2]),
               "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7])
               : "memory");
}
__device__ __forceinline__ uint4 ld16_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <typename GT> struct Grad;
template <> struct Grad<float> {
  static __device__ __forceinline__ void load8(const float* p, float (&g)[8]) { ld8_stream(p, g); }
  static __device__ __forceinline__ float load1(const float* p) { return __ldg(p); }
};
template <> struct Grad<__half> {
  static __device__ __forceinline__ void load8(const __half* p, float (&g)[8]) {
    const uint4 u = ld16_stream(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
      g[2 * k] = f.x;
      g[2 * k + 1] = f.y;
    }
  }
  static __device__ __forceinline__ float load1(const __half* p) { return __half2float(__ldg(p)); }
};
template <> struct Grad<__nv_bfloat16> {
  static __device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&g)[8]) {
    const uint4 u = ld16_stream(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      g[2 * k] = __uint_as_float(w[k] << 16);
      g[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  }
  static __device__ __forceinline__ float load1(const __nv_bfloat16* p) { return __bfloat162float(__ldg(p)); }
};

// ------------------------------------------------------------------------------------------------
// fixed-order CTA reduction of one double per thread

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int NT>
__device__ __forceinline__ double block_sum(double v, double* red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    r = lane < NT / 32 ? red[lane] : 0.0;
    r = warp_sum(r);
  }
  __syncthreads();
  return r;  // valid in thread 0
}

// Sum of squares without rounding error at the element level: c*c = p + pe exactly (FMA), p is
// added to the running fp32 sum with an exact two-sum, and the two error terms are collected in a
// second fp32 word.  (hi, lo) carries ~44 bits; the block sums the pairs as pairs (below) and promotes
// one total to double per work unit.  This
// keeps the scales equal to a double-precision evaluation (1 ulp at most, almost always 0) without
// using the GPU's slow fp64 pipe per element.  Written with Blackwell's packed fp32x2 arithmetic for
// two elements at once: (hi, lo) hold two independent (hi, lo) accumulators, one per half.
__device__ __forceinline__ void add_square2(unsigned long long& hi, unsigned long long& lo, float c0, float c1) {
  asm("{\n\t.reg .b64 c, p, np, pe, s, bb, t, u, e;\n\t"
      "mov.b64 c, {%2, %3};\n\t"
      "mul.rn.f32x2 p, c, c;\n\t"
      "xor.b64 np, p, 0x8000000080000000;\n\t"
      "fma.rn.f32x2 pe, c, c, np;\n\t"
      "add.rn.f32x2 s, %0, p;\n\t"
      "sub.rn.f32x2 bb, s, %0;\n\t"
      "sub.rn.f32x2 t, s, bb;\n\t"
      "sub.rn.f32x2 t, %0, t;\n\t"
      "sub.rn.f32x2 u, p, bb;\n\t"
      "add.rn.f32x2 e, t, u;\n\t"
      "add.rn.f32x2 e, e, pe;\n\t"
      "add.rn.f32x2 %1, %1, e;\n\t"
      "mov.b64 %0, s;\n\t}"
      : "+l"(hi), "+l"(lo)
      : "f"(c0), "f"(c1));
}

// The threads' (hi, lo) accumulators are summed across the block as fp32 pairs too: s + e, where s
// takes each addition's rounded sum and e collects its exact rounding error (two-sum) along with the
// error words.  Only the block's final pair is promoted to double, once per unit: the GPU's fp64
// pipe is slow (about two operations per clock and SM), and a double reduction over every thread
// held it for over a thousand cycles per unit.  Each pair addition is symmetric in its operands, so
// the butterfly leaves the same value in every lane; e's own roundings stay below 2^-40 of the total.
struct SqPair {
  float s, e;
};
__device__ __forceinline__ SqPair sq_add(SqPair a, SqPair b) {
  const float s = __fadd_rn(a.s, b.s);
  const float bb = __fsub_rn(s, a.s);
  const float err = __fadd_rn(__fsub_rn(a.s, __fsub_rn(s, bb)), __fsub_rn(b.s, bb));  // a.s + b.s - s, exactly
  return {s, __fadd_rn(__fadd_rn(a.e, b.e), err)};
}
// this thread's two (hi, lo) halves as one pair
__device__ __forceinline__ SqPair sq_of(unsigned long long hi, unsigned long long lo) {
  return sq_add({__uint_as_float((uint32_t)hi), __uint_as_float((uint32_t)lo)},
                {__uint_as_float((uint32_t)(hi >> 32)), __uint_as_float((uint32_t)(lo >> 32))});
}
// butterfly over the first W lanes of the warp (W a power of two; the others hold zeros or are ignored)
template <int W>
__device__ __forceinline__ SqPair warp_sq(SqPair p) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1)
    p = sq_add(p, {__shfl_xor_sync(0xffffffffu, p.s, o), __shfl_xor_sync(0xffffffffu, p.e, o)});
  return p;
}
__device__ __forceinline__ double sq_value(SqPair p) { return (double)p.s + (double)p.e; }

// Fixed-order block total of the threads' pairs: the warps' butterflies, then warp 0 over the warp
// totals (red: NT/32 slots of 8 bytes at least).  In thread 0 (block_sq) or every thread
// (block_sq_all, red: NT/32 + 1 slots).
template <int NT>
__device__ __forceinline__ double block_sq(SqPair p, double* red) {
  static_assert(NT % 32 == 0 && ((NT / 32) & (NT / 32 - 1)) == 0, "a power-of-two number of warps");
  float2* r2 = reinterpret_cast<float2*>(red);
  p = warp_sq<32>(p);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) r2[warp] = make_float2(p.s, p.e);
  __syncthreads();
  double r = 0.0;
  if (warp == 0) {
    const float2 v = lane < NT / 32 ? r2[lane] : make_float2(0.0f, 0.0f);
    r = sq_value(warp_sq<NT / 32>({v.x, v.y}));
  }
  __syncthreads();
  return r;
}
template <int NT>
__device__ __forceinline__ double block_sq_all(SqPair p, double* red) {
  const double r = block_sq<NT>(p, red);
  if (threadIdx.x == 0) red[NT / 32] = r;
  __syncthreads();
  return red[NT / 32];
}

// Range of the fp32-pair accumulation.  Each square is exact for |c| >= 2^-51 (below that its
// rounding residual falls off fp32's subnormal grid, and below 2^-75 the square itself is lost), and
// a thread's running sum cannot overflow while the unit's total stays far below 2^128.  A unit whose
// total lies outside [kSquaresLo, kSquaresHi) -- all of its values tiny, values near overflow, or a
// non-finite value -- is summed again from its stored values in double, where every square is
// exact, so the scales follow the exact sum at any magnitude.  Inside the range, squares that lost
// bits (each below 2^-102, at most 2^16 of them in a unit) move a total of at least 2^-56 by less
// than 2^-30 of itself.  Normal workloads never leave the range: the check costs one comparison per
// unit.
constexpr double kSquaresLo = 0x1p-56;
constexpr double kSquaresHi = 0x1p100;
__device__ __forceinline__ bool squares_inexact(double tot) { return !(tot >= kSquaresLo && tot < kSquaresHi); }

// This thread's share (elements tid, tid + nt, ...) of the sum of squares of v[0, len) in double,
// read through L2 (the values were written by other threads of the block before a barrier).
__device__ __forceinline__ double squares_fp64(const float* v, int len, int tid, int nt) {
  double s = 0.0;
  for (int e = tid; e < len; e += nt) {
    const double x = (double)__ldcg(v + e);
    s = __dadd_rn(s, __dmul_rn(x, x));
  }
  return s;
}

// The rare fp64 path: warp 0 sums the unit's stored values again (a fixed order: lane l takes
// elements l, l + 32, ...) and the block receives the total through red[NT/32 + 1].
template <int NT>
__device__ __forceinline__ double unit_squares_fp64(const float* v, int len, double* red) {
  if (threadIdx.x < 32) {
    const double s = warp_sum(squares_fp64(v, len, threadIdx.x, 32));
    if (threadIdx.x == 0) red[NT / 32 + 1] = s;
  }
  __syncthreads();
  return red[NT / 32 + 1];
}

// A unit's sum of squares for the whole block (every thread calls it and receives the result): the
// fp32-pair total, or the fp64 sum of the unit's stored values v[0, len) when that total is outside
// the exact range.  red: NT/32 + 2 slots.
template <int NT>
__device__ __forceinline__ double unit_squares(unsigned long long hi, unsigned long long lo, const float* v, int len,
                                               double* red) {
  const double tot = block_sq_all<NT>(sq_of(hi, lo), red);
  return squares_inexact(tot) ? unit_squares_fp64<NT>(v, len, red) : tot;
}

// Transpose of an 8x8 bit matrix held in a 64-bit word (bit 8r+c -> bit 8c+r), by three rounds of
// masked bit swaps (the classic recursive block transpose).
__device__ __forceinline__ uint64_t transpose8x8(uint64_t x) {
  uint64_t t;
  t = (x ^ (x >> 7)) & 0x00AA00AA00AA00AAull;
  x = x ^ t ^ (t << 7);
  t = (x ^ (x >> 14)) & 0x0000CCCC0000CCCCull;
  x = x ^ t ^ (t << 14);
  t = (x ^ (x >> 28)) & 0x00000000F0F0F0F0ull;
  x = x ^ t ^ (t << 28);
  return x;
}

// +s when the bit is set, -s otherwise (flip of the sign bit)
__device__ __forceinline__ float signed_scale(float s, uint32_t byte, int q) {
  return __int_as_float(__float_as_int(s) ^ ((~byte << (31 - q)) & 0x80000000u));
}

// the fp32 operations of the method, in the oracle's order
__device__ __forceinline__ float momentum(float b1, float omb1, float m, float g) {
  return __fadd_rn(__fmul_rn(b1, m), __fmul_rn(omb1, g));
}
__device__ __forceinline__ float error_of(float c, float s) {  // c - s*sign(c), sign(0) = +1
  return c >= 0.0f ? __fsub_rn(c, s) : __fadd_rn(c, s);
}

// ------------------------------------------------------------------------------------------------
// K1: worker momentum + error feedback + 1-bit compression + norm partials.
// One unit = (worker-side chunk, worker).  c_i = (b1*m + (1-b1)*g_i) + delta_i, delta_i rebuilt
// from the previous c_i and s_i; writes c_i, its sign byte and the chunk's sum of c_i^2.

// Where the worker kernel's momentum comes from.
enum MomentumSource : int {
  kMomBits = 0,        // the previous broadcast: S * sign(a), from the server sign bits
  kMomDense = 1,       // the fp32 buffer (first compression step, after an import)
  kMomNone = 2,        // no momentum: c_i = g_i + delta_i (the gradient-compression baseline)
  kMomBitsShards = 3   // as kMomBits, for plans whose worker chunks may hold several shards
};

// WU: one warp per unit instead of one block (plans whose worker chunks are all short, at most
// kWarpUnitMax elements): eight units per block, and each unit's sum of squares is a warp butterfly,
// with no block barrier per unit.
constexpr int kWarpUnitMax = 8192;

template <typename GT, int MSRC, bool HAS_ERR, bool VEC, bool WU = false>
__global__ void __launch_bounds__(kThreads) k_worker(const StepArgs A) {
  constexpr bool DENSE_M = MSRC == kMomDense;
  constexpr bool BITS = MSRC == kMomBits || MSRC == kMomBitsShards;
  __shared__ double red[kThreads / 32];
  const int64_t n_units = (int64_t)A.n_wchunks * A.nl;
  for (int64_t u = WU ? (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5) : (int64_t)blockIdx.x;
       u < n_units; u += WU ? (int64_t)gridDim.x * (kThreads / 32) : (int64_t)gridDim.x) {
    const int ci = (int)(u / A.nl);
    const int il = (int)(u - (int64_t)ci * A.nl);  // local worker; global worker i
    const int i = A.w0 + il;
    const Chunk ch = A.wchunks[ci];
    ONEBIT_CHECK_UNIT(worker_unit_ok(A, ch, il), A.status, ONEBIT_K_WORKER)
    const GT* __restrict__ g = static_cast<const GT*>(A.gptr[(int64_t)il * A.T + ch.seg]) + ch.start;
    float* __restrict__ c = A.c + (int64_t)il * A.Dp + ch.off;
    uint8_t* __restrict__ wb = reinterpret_cast<uint8_t*>(A.wbits + (int64_t)i * A.Wr) + (ch.off >> 3);
    const uint8_t* __restrict__ sb = reinterpret_cast<const uint8_t*>(A.sbits) + (ch.off >> 3);
    const float* __restrict__ md = A.m + ch.off;
    const float sp = HAS_ERR ? A.wscale_prev[(int64_t)i * A.T + ch.seg] : 0.0f;
    const float Sp = BITS ? A.sscale_prev[(int64_t)ch.seg * A.n + ch.shard] : 0.0f;
    const float b1 = A.b1, omb1 = A.omb1;
    // a chunk that holds several whole server shards (short shards only) takes each group's broadcast
    // scale from that group's own shard: shard + (offset inside the chunk) / shard length
    const float* __restrict__ Sseg = A.sscale_prev + (int64_t)ch.seg * A.n + ch.shard;
    auto scale_of = [&](int gi) { return ch.per ? Sseg[(uint32_t)(gi * 8) / (uint32_t)ch.per] : Sp; };

    // one group of 8 elements: loads first (so that two groups are in flight), then math + stores
    struct In {
      float g[8], cp[8], m[8];
      uint32_t mb;
      float S;
    };
    (void)DENSE_M;
    auto load = [&](In& r, int gi) {
      const int64_t e = (int64_t)gi * 8;
      if (VEC) {
        Grad<GT>::load8(g + e, r.g);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) r.g[q] = Grad<GT>::load1(g + e + q);
      }
      if (HAS_ERR) ld8_state(c + e, r.cp);
      if (MSRC == kMomDense) ld8_stream(md + e, r.m);
      if (BITS) r.mb = sb[gi];
      if (MSRC == kMomBitsShards) r.S = scale_of(gi);
    };
    unsigned long long hi = 0, lo = 0;  // this thread's sum of c^2 over the unit (two lanes)
    auto work = [&](const In& r, int gi) {
      float out[8];
      uint32_t byte = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float mi;
        if (MSRC == kMomNone) {
          mi = r.g[q];
        } else {
          const float Sg = MSRC == kMomBitsShards ? r.S : Sp;
          const float mq = MSRC == kMomDense ? r.m[q] : (((r.mb >> q) & 1u) ? Sg : -Sg);
          mi = momentum(b1, omb1, mq, r.g[q]);
        }
        const float d = HAS_ERR ? error_of(r.cp[q], sp) : 0.0f;
        const float cq = __fadd_rn(mi, d);
        out[q] = cq;
        byte |= (cq >= 0.0f ? 1u : 0u) << q;
      }
#pragma unroll
      for (int q = 0; q < 8; q += 2) add_square2(hi, lo, out[q], out[q + 1]);
      st8(c + (int64_t)gi * 8, out);
      wb[gi] = (uint8_t)byte;
    };

    const int ng = ch.len >> 3;
    constexpr int NT = WU ? 32 : kThreads;  // threads sharing the unit
    int gi = WU ? (int)(threadIdx.x & 31) : (int)threadIdx.x;
    for (; gi + (kWorkerUnroll - 1) * NT < ng; gi += kWorkerUnroll * NT) {
      In r[kWorkerUnroll];  // all loads of kWorkerUnroll groups in flight, then the math
#pragma unroll
      for (int j = 0; j < kWorkerUnroll; ++j) load(r[j], gi + j * NT);
#pragma unroll
      for (int j = 0; j < kWorkerUnroll; ++j) work(r[j], gi + j * NT);
    }
    for (; gi < ng; gi += NT) {
      In r0;
      load(r0, gi);
      work(r0, gi);
    }
    const int rem = ch.len & 7;
    if (rem && (WU ? (int)(threadIdx.x & 31) : (int)threadIdx.x) == (ng % NT)) {  // the ragged end of a tensor: scalar
      const int64_t e0 = (int64_t)ng * 8;
      const float St = MSRC == kMomBitsShards ? scale_of(ng) : Sp;
      uint32_t byte = 0;
      for (int q = 0; q < rem; ++q) {
        const int64_t e = e0 + q;
        float mi;
        if (MSRC == kMomNone) {
          mi = Grad<GT>::load1(g + e);
        } else {
          const float mq = MSRC == kMomDense ? md[e] : (((sb[ng] >> q) & 1u) ? St : -St);
          mi = momentum(b1, omb1, mq, Grad<GT>::load1(g + e));
        }
        const float d = HAS_ERR ? error_of(c[e], sp) : 0.0f;
        const float cq = __fadd_rn(mi, d);
        c[e] = cq;
        byte |= (cq >= 0.0f ? 1u : 0u) << q;
        add_square2(hi, lo, cq, 0.0f);
      }
      wb[ng] = (uint8_t)byte;
    }
    if (WU) {
      const double tot = sq_value(warp_sq<32>(sq_of(hi, lo)));
      if ((threadIdx.x & 31) == 0) A.wpart[(int64_t)il * A.n_wchunks + ci] = tot;
    } else {
      const double tot = block_sq<kThreads>(sq_of(hi, lo), red);
      if (threadIdx.x == 0) A.wpart[(int64_t)il * A.n_wchunks + ci] = tot;
    }
  }
}

// Exact-range repair of the worker partials.  A unit whose fast total lies outside the exact range of
// the fp32-pair squares (all its values tiny, or near overflow) is summed again in double from its
// stored c.  One thread per unit scans the partials; the units found are recomputed by the whole
// block, each in a fixed order, so the result does not depend on which block finds them.  Kept out of
// k_worker, whose streaming loop stays free of this rare code.
static __global__ void __launch_bounds__(kThreads) k_worker_exact(const StepArgs A) {
  __shared__ double red[kThreads / 32 + 2];
  __shared__ int n_found;
  __shared__ int found[kThreads];
  const int64_t n_parts = (int64_t)A.nl * A.n_wchunks;  // partial il*n_wchunks + ci: local worker il, chunk ci
  for (int64_t base = (int64_t)blockIdx.x * kThreads; base < n_parts; base += (int64_t)gridDim.x * kThreads) {
    if (threadIdx.x == 0) n_found = 0;
    __syncthreads();
    const int64_t q = base + threadIdx.x;
    if (q < n_parts && squares_inexact(__ldcg(A.wpart + q))) found[atomicAdd(&n_found, 1)] = threadIdx.x;
    __syncthreads();
    for (int f = 0; f < n_found; ++f) {
      const int64_t qq = base + found[f];
      const int il = (int)(qq / A.n_wchunks), ci = (int)(qq - (int64_t)il * A.n_wchunks);
      const Chunk ch = A.wchunks[ci];
      ONEBIT_CHECK_UNIT(worker_unit_ok(A, ch, il), A.status, ONEBIT_K_WORKER_SCALE)
      const double tot = unit_squares_fp64<kThreads>(A.c + (int64_t)il * A.Dp + ch.off, ch.len, red);
      if (threadIdx.x == 0) A.wpart[qq] = tot;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------------
// Scale kernels: one CTA per (worker, tensor) or (tensor, shard); fixed-order sum of the chunk
// partials, then scale = sqrt(sum / len) in double, rounded once to fp32.

__device__ __forceinline__ float finish_scale(const double* part, const Range r, unsigned int* status,
                                              double* red) {
  double acc = 0.0;
  for (int c = threadIdx.x; c < r.count; c += kScaleThreads) acc += __ldcg(part + r.first + c);
  const double tot = block_sum<kScaleThreads>(acc, red);
  float s = 0.0f;
  if (threadIdx.x == 0) {
    s = r.len > 0 ? __double2float_rn(sqrt(tot / (double)r.len)) : 0.0f;
    if (!isfinite(s)) atomicOr(status, 1u);
  }
  return s;
}

// one scale per (local worker, tensor): item = il*T + k, written to global worker w0 + il
static __global__ void __launch_bounds__(kScaleThreads) k_worker_scale(const StepArgs A) {
  __shared__ double red[kScaleThreads / 32];
  const int il = blockIdx.x / A.T, k = blockIdx.x % A.T;
  ONEBIT_CHECK_ITEM(range_ok(A.wseg_ranges[k], A.n_wchunks) && il < A.nl && A.w0 + il < A.n, A.status,
                    ONEBIT_K_WORKER_SCALE)
  const float s = finish_scale(A.wpart + (int64_t)il * A.n_wchunks, A.wseg_ranges[k], A.status, red);
  if (threadIdx.x == 0) A.wscale_cur[(int64_t)A.w0 * A.T + blockIdx.x] = s;
}

static __global__ void __launch_bounds__(kScaleThreads) k_server_scale(const StepArgs A) {
  __shared__ double red[kScaleThreads / 32];
  ONEBIT_CHECK_ITEM(range_ok(A.shard_ranges[blockIdx.x], A.n_chunks) && (int)blockIdx.x < A.n * A.T, A.status,
                    ONEBIT_K_SERVER_SCALE)
  const float s = finish_scale(A.spart, A.shard_ranges[blockIdx.x], A.status, red);
  if (threadIdx.x == 0) A.sscale_cur[blockIdx.x] = s;
}

// The same sums for lists of many short ranges (at most kWarpScaleMax partials each): one warp per
// scale, kScaleThreads/32 scales per CTA.  A plan uses one form or the other for all its scales of a
// kind, so the summation order is fixed for a given plan.
constexpr int kWarpScaleMax = 256;
__device__ __forceinline__ float finish_scale_warp(const double* part, const Range r, unsigned int* status) {
  const int lane = threadIdx.x & 31;
  double acc = 0.0;
  for (int c = lane; c < r.count; c += 32) acc += __ldcg(part + r.first + c);
  acc = warp_sum(acc);
  float s = 0.0f;
  if (lane == 0) {
    s = r.len > 0 ? __double2float_rn(sqrt(acc / (double)r.len)) : 0.0f;
    if (!isfinite(s)) atomicOr(status, 1u);
  }
  return s;
}

static __global__ void __launch_bounds__(kScaleThreads) k_worker_scale_warp(const StepArgs A) {
  const int item = blockIdx.x * (kScaleThreads / 32) + (threadIdx.x >> 5);
  if (item >= A.nl * A.T) return;  // the whole warp
  const int il = item / A.T, k = item % A.T;
  ONEBIT_CHECK_ITEM(range_ok(A.wseg_ranges[k], A.n_wchunks) && A.w0 + il < A.n, A.status, ONEBIT_K_WORKER_SCALE)
  const float s = finish_scale_warp(A.wpart + (int64_t)il * A.n_wchunks, A.wseg_ranges[k], A.status);
  if ((threadIdx.x & 31) == 0) A.wscale_cur[(int64_t)A.w0 * A.T + item] = s;
}

static __global__ void __launch_bounds__(kScaleThreads) k_server_scale_warp(const StepArgs A) {
  const int item = blockIdx.x * (kScaleThreads / 32) + (threadIdx.x >> 5);
  if (item >= A.n * A.T) return;
  ONEBIT_CHECK_ITEM(range_ok(A.shard_ranges[item], A.n_chunks), A.status, ONEBIT_K_SERVER_SCALE)
  const float s = finish_scale_warp(A.spart, A.shard_ranges[item], A.status);
  if ((threadIdx.x & 31) == 0) A.sscale_cur[item] = s;
}

// Plans whose every range holds at most one partial (short scale blocks: one chunk per shard or per
// block): one thread per scale.  The sum of a single partial involves no rounding, so the scales equal
// the warp form's bit for bit, at a 32nd of its fp64 instructions (GB300's fp64 pipe is slow).
__device__ __forceinline__ float scale_of_one(const double* part, const Range r, unsigned int* status) {
  const double tot = r.count > 0 ? __ldcg(part + r.first) : 0.0;
  const float s = r.len > 0 ? __double2float_rn(sqrt(tot / (double)r.len)) : 0.0f;
  if (!isfinite(s)) atomicOr(status, 1u);
  return s;
}

static __global__ void __launch_bounds__(kScaleThreads) k_worker_scale_one(const StepArgs A) {
  const int item = blockIdx.x * kScaleThreads + threadIdx.x;
  if (item >= A.nl * A.T) return;
  const int il = item / A.T, k = item % A.T;
  ONEBIT_CHECK_ITEM(range_ok(A.wseg_ranges[k], A.n_wchunks) && A.wseg_ranges[k].count <= 1 && A.w0 + il < A.n,
                    A.status, ONEBIT_K_WORKER_SCALE)
  A.wscale_cur[(int64_t)A.w0 * A.T + item] =
      scale_of_one(A.wpart + (int64_t)il * A.n_wchunks, A.wseg_ranges[k], A.status);
}

static __global__ void __launch_bounds__(kScaleThreads) k_server_scale_one(const StepArgs A) {
  const int item = blockIdx.x * kScaleThreads + threadIdx.x;
  if (item >= A.n * A.T) return;
  ONEBIT_CHECK_ITEM(range_ok(A.shard_ranges[item], A.n_chunks) && A.shard_ranges[item].count <= 1, A.status,
                    ONEBIT_K_SERVER_SCALE)
  A.sscale_cur[item] = scale_of_one(A.spart, A.shard_ranges[item], A.status);
}

// ------------------------------------------------------------------------------------------------
// K2: server.  For every element the n decompressed worker messages are summed in worker order in
// fp32, divided by n, and the server error is added; the result a is written with its sign byte, and
// each chunk's sum of a^2 is kept.
//
// The ordered sum over the first min(n, 12) workers depends only on their 12 sign bits, so it is read
// from a 4096-entry shared-memory table built per tensor with exactly those fp32 additions
// (level k: T_k[p] = T_{k-1}[p mod 2^k] + (bit k of p ? s_k : -s_k), starting from 0 + x_0).
// Two 8x8 bit transposes turn the workers' sign bytes into the 8 elements' table indices.  Workers
// 12..15 are then added one by one in order; their four signed scales come as one float4 from a
// 16-entry table indexed by their 4 sign bits (one copy per lane, so the lookups never conflict).
// Workers 16.. (if any) are added from their sign bytes.  The result is the same fp32 value as the
// plain left-to-right sum.

constexpr int kLutBits = 12;  // workers folded into the server's sum table

struct ServerTables {
  float ssc[kMaxWorkers];
  float lut[1 << kLutBits];
  float4 quad[16 * 32];  // [pattern of workers 12..15][lane]
  double red[kThreads / 32 + 2];
};

// Rebuild the tables for tensor `seg` (block-wide; every thread calls it).
__device__ __forceinline__ void build_server_tables(ServerTables& S, const StepArgs& A, int seg) {
  const int n = A.n, nl = n < kLutBits ? n : kLutBits;
  __syncthreads();  // everyone is done with the previous tables
  for (int i = threadIdx.x; i < n; i += kThreads) S.ssc[i] = A.wscale_cur[(int64_t)i * A.T + seg];
  __syncthreads();
  if (threadIdx.x == 0) {
    S.lut[0] = __fadd_rn(0.0f, -S.ssc[0]);
    S.lut[1] = __fadd_rn(0.0f, S.ssc[0]);
  }
  __syncthreads();
  for (int k = 1; k < nl; ++k) {
    const float sk = S.ssc[k];
    for (int p = threadIdx.x; p < (1 << k); p += kThreads) {
      const float old = S.lut[p];
      S.lut[p] = __fadd_rn(old, -sk);
      S.lut[p + (1 << k)] = __fadd_rn(old, sk);
    }
    __syncthreads();
  }
  if (n > kLutBits) {
    for (int p = threadIdx.x; p < 16 * 32; p += kThreads) {
      const int pat = p >> 5;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float sj = kLutBits + j < n ? S.ssc[kLutBits + j] : 0.0f;
        v[j] = ((pat >> j) & 1) ? sj : -sj;
      }
      S.quad[p] = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
  }
}

// Ordered sum of the first min(n, 16) workers' decompressed messages for 8 elements, from their sign
// bytes b[0..15] (bytes of absent workers are 0).
__device__ __forceinline__ uint32_t pack4(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3) {
  return __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);  // b0 | b1<<8 | ...
}

// PTX byte permute in its default mode: each selector nibble's low 3 bits pick one of the 8 source
// bytes, and a set top bit replicates that byte's sign bit over the whole result byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ void server_sum16(const ServerTables& S, int n, const uint32_t (&b)[16], float (&s)[8]) {
  const int lane = threadIdx.x & 31;
  const uint64_t t0 = transpose8x8(((uint64_t)pack4(b[4], b[5], b[6], b[7]) << 32) | pack4(b[0], b[1], b[2], b[3]));
  uint64_t t1 = 0;
  if (n > 8) t1 = transpose8x8(((uint64_t)pack4(b[12], b[13], b[14], b[15]) << 32) | pack4(b[8], b[9], b[10], b[11]));
  // byte q of t0: workers 0..7 of element q; of t1: workers 8..15.  Split t1 into workers 8..11 (low
  // nibbles, mid) and 12..15 (hi), so that one byte permute yields each element's table index.
  const uint32_t t0w[2] = {(uint32_t)t0, (uint32_t)(t0 >> 32)};
  const uint32_t mid[2] = {(uint32_t)t1 & 0x0f0f0f0fu, (uint32_t)(t1 >> 32) & 0x0f0f0f0fu};
  const uint32_t hiw[2] = {((uint32_t)t1 >> 4) & 0x0f0f0f0fu, ((uint32_t)(t1 >> 32) >> 4) & 0x0f0f0f0fu};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    // index bits 0..7: workers 0..7, bits 8..11: workers 8..11; bytes 2-3 are the sign replica of a
    // byte of mid (whose top bit is 0), i.e. zero
    const uint32_t r = (q & 3) + 4;
    const uint32_t x = prmt(t0w[q >> 2], mid[q >> 2], (q & 3) | (r << 4) | ((8 | r) << 8) | ((8 | r) << 12));
    s[q] = S.lut[x];
    if (n > kLutBits) {  // workers 12..15, in order
      const uint32_t pat = __byte_perm(hiw[q >> 2], 0u, (q & 3) | 0x4440u);
      const float4 qv = S.quad[pat * 32 + lane];
      s[q] = __fadd_rn(s[q], qv.x);
      if (n > kLutBits + 1) s[q] = __fadd_rn(s[q], qv.y);
      if (n > kLutBits + 2) s[q] = __fadd_rn(s[q], qv.z);
      if (n > kLutBits + 3) s[q] = __fadd_rn(s[q], qv.w);
    }
  }
}

__device__ __forceinline__ void server_add_worker(float (&s)[8], float si, uint32_t byte) {
#pragma unroll
  for (int q = 0; q < 8; ++q) s[q] = __fadd_rn(s[q], signed_scale(si, byte, q));
}

// a = sum / n + eps_prev, its sign byte (bits past `cnt` cleared) and the squares of the first cnt.
// NW > 0: the worker count is the compile-time constant NW (the same arithmetic, folded).
template <bool HAS_ERR, int NW = 0>
__device__ __forceinline__ uint32_t server_finish(const StepArgs& A, const float (&s)[8], const float (&ap)[8],
                                                  float Sp, int cnt, float (&out)[8], unsigned long long& hi,
                                                  unsigned long long& lo) {
  constexpr bool kPow2 = NW > 0 && (NW & (NW - 1)) == 0;
  uint32_t byte = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    // x / n, as x * (1/n) when n is a power of two (bit-identical); 1/n is exact there
    const float avg = NW > 0 ? (kPow2 ? __fmul_rn(s[q], 1.0f / NW) : __fdiv_rn(s[q], (float)NW))
                             : (A.pow2 ? __fmul_rn(s[q], A.inv_n) : __fdiv_rn(s[q], A.nf));
    // the server error a - Sp*sign(a), as a - copysign(Sp, a): the same value except for a = -0, which a
    // kernel never stores (the sum is never -0) and an import stores only with Sp = 0, where either
    // form gives a zero and avg + ep is unchanged
    const float ep = HAS_ERR ? __fsub_rn(ap[q], copysignf(Sp, ap[q])) : 0.0f;
    out[q] = __fadd_rn(avg, ep);
    byte |= (out[q] >= 0.0f ? 1u : 0u) << q;
  }
  if (cnt >= 8) {
#pragma unroll
    for (int q = 0; q < 8; q += 2) add_square2(hi, lo, out[q], out[q + 1]);
  } else {
    byte &= (1u << cnt) - 1u;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < cnt) add_square2(hi, lo, out[q], 0.0f);
  }
  return byte;
}

__device__ __forceinline__ void store_a(float* a, int64_t e, int cnt, const float (&out)[8]) {
  if (cnt >= 8) {
    st8(a + e, out);
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < cnt) a[e + q] = out[q];
  }
}

// Which chunks a server CTA takes.  Normally every gridDim.x-th chunk.  For lists of many short
// tensors or scale blocks (CONTIG) one contiguous run instead, so that consecutive chunks of a
// segment share one CTA and its sum tables are rebuilt once per segment and CTA, not once per chunk;
// the runs split the elements evenly (the first chunk whose element offset reaches b*D/gridDim.x).
__device__ __forceinline__ int run_begin(const StepArgs& A, int b) {
  if (b >= (int)gridDim.x) return A.n_chunks;
  const int64_t target = b * A.D / gridDim.x;
  int lo = 0, hi = A.n_chunks;  // first chunk with uoff >= target
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (A.chunks[mid].uoff < target) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}


// K2, register variant (any n; launched for n > 128, where the staged ring no longer fits): every
// thread loads its group's sign bytes and a directly.
template <bool HAS_ERR, bool CONTIG>
__global__ void __launch_bounds__(kThreads) k_server(const StepArgs A) {
  __shared__ ServerTables S;
  const int n = A.n;
  const int64_t wrow = A.Wr * 4;  // bytes per worker row of sign words
  int cur_seg = -1;
  int u_begin = blockIdx.x, u_end = A.n_chunks, u_step = gridDim.x;
  if constexpr (CONTIG) {
    u_begin = run_begin(A, blockIdx.x);
    u_end = run_begin(A, blockIdx.x + 1);
    u_step = 1;
  }
  for (int u = u_begin; u < u_end; u += u_step) {
    const Chunk ch = A.chunks[u];
    ONEBIT_CHECK_UNIT(chunk_ok(A, ch), A.status, ONEBIT_K_SERVER)
    if (ch.seg != cur_seg) {  // block-uniform
      build_server_tables(S, A, ch.seg);
      cur_seg = ch.seg;
    }
    const float Sp = HAS_ERR ? A.sscale_prev[(int64_t)ch.seg * n + ch.shard] : 0.0f;
    float* __restrict__ a = A.a + ch.off;
    const uint8_t* __restrict__ wb = reinterpret_cast<const uint8_t*>(A.wbits) + (ch.off >> 3);
    uint8_t* __restrict__ sb = reinterpret_cast<uint8_t*>(A.sbits) + (ch.off >> 3);
    unsigned long long hi = 0, lo = 0;
    const int ng = (ch.len + 7) >> 3;
    for (int gi = threadIdx.x; gi < ng; gi += kThreads) {
      const int64_t e = (int64_t)gi * 8;
      const int cnt = ch.len - gi * 8;  // >= 8 except in a tensor's last group
      uint32_t b[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] = i < n ? (uint32_t)__ldg(wb + (int64_t)i * wrow + gi) : 0u;
      float ap[8];
      if (HAS_ERR) {
        if (cnt >= 8) {
          ld8_state(a + e, ap);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) ap[q] = q < cnt ? a[e + q] : 0.0f;
        }
      }
      float sum[8];
      server_sum16(S, n, b, sum);
      for (int i = 16; i < n; ++i) server_add_worker(sum, S.ssc[i], __ldg(wb + (int64_t)i * wrow + gi));
      float out[8];
      const uint32_t byte = server_finish<HAS_ERR>(A, sum, ap, Sp, cnt, out, hi, lo);
      store_a(a, e, cnt, out);
      sb[gi] = (uint8_t)byte;
    }
    const double tot = unit_squares<kThreads>(hi, lo, a, ch.len, S.red);
    if (threadIdx.x == 0) A.spart[u] = tot;
  }
}

// ------------------------------------------------------------------------------------------------
// K2, staged variant (n <= kStageMaxWorkers), warp-specialised.  A ring of kStages shared-memory
// stages each holds one tile of kTile elements of a and the n workers' sign bytes for it.  One
// producer warp keeps the ring full with bulk asynchronous copies (cp.async.bulk; completion counted
// on a "full" mbarrier per stage); kConsumerWarps consumer warps compute from shared memory and
// release a stage by arriving on its "empty" mbarrier.  Consumers synchronise with each other only
// through a named barrier, when the tables are rebuilt and at the end of each chunk.
//
// Every wait is bounded (kWaitCycles, about one second).  A wait that runs out sets status bit 2 and
// the block-wide abort flag; from then on every thread skips its waits and its work but keeps
// stepping through the same sequence, so that the named barriers still meet, and the producer drains
// its own copies still in flight (bounded again) before the block ends.

constexpr int kTile = 4096;                 // elements per tile (two groups per consumer thread)
constexpr int kStages = 2;                 // two stages leave room for three CTAs per SM
constexpr int kStageMaxWorkers = 128;         // two stages of n sign rows + a still fit (one CTA per SM at 128)
constexpr int kRowBytes = kTile / 8 + 32;   // a 16-byte aligned window around the tile's sign bytes
constexpr int kConsumerWarps = kThreads / 32;
constexpr int kStagedThreads = kThreads + 32;      // consumers + one producer warp
constexpr long long kWaitCycles = 2000000000LL;    // ~1 s at the maximum SM clock

__host__ __device__ constexpr size_t server_stage_bytes(int n) { return (size_t)kTile * 4 + (size_t)n * kRowBytes; }
__host__ __device__ constexpr size_t server_dyn_smem(int n) { return kStages * server_stage_bytes(n) + 2 * kStages * 8; }

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// bounded wait: false if the phase did not complete within kWaitCycles
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kThreads) : "memory"); }

// The consumer warps' fixed-order total of the consumer threads' squares (the pair reduction of
// block_sq), left in red[kConsumerWarps] (red: kConsumerWarps + 1 slots at least).  *redo is set when
// that total lies outside the exact range of the fp32-pair squares and the block has not aborted.
__device__ __forceinline__ void consumers_total(SqPair p, double* red, int* redo, const volatile int* abort) {
  static_assert((kConsumerWarps & (kConsumerWarps - 1)) == 0, "a power-of-two number of consumer warps");
  float2* r2 = reinterpret_cast<float2*>(red);
  p = warp_sq<32>(p);
  if ((threadIdx.x & 31) == 0) r2[threadIdx.x >> 5] = make_float2(p.s, p.e);
  consumers_sync();
  if (threadIdx.x < 32) {
    const float2 v = threadIdx.x < kConsumerWarps ? r2[threadIdx.x] : make_float2(0.0f, 0.0f);
    const double r = sq_value(warp_sq<kConsumerWarps>({v.x, v.y}));
    if (threadIdx.x == 0) {
      red[kConsumerWarps] = r;
      *redo = squares_inexact(r) && !*abort;
    }
  }
  consumers_sync();
}

struct TileCursor {  // position in this block's sequence of (unit, tile)
  int u, t;
};

__device__ __forceinline__ int tiles_of(const Chunk& ch) { return (ch.len + kTile - 1) / kTile; }

// table rebuild among the consumer threads only (same arithmetic as build_server_tables)
__device__ __forceinline__ void build_server_tables_consumers(ServerTables& S, const StepArgs& A, int seg) {
  const int n = A.n, nl = n < kLutBits ? n : kLutBits;
  consumers_sync();
  for (int i = threadIdx.x; i < n; i += kThreads) S.ssc[i] = A.wscale_cur[(int64_t)i * A.T + seg];
  consumers_sync();
  if (threadIdx.x == 0) {
    S.lut[0] = __fadd_rn(0.0f, -S.ssc[0]);
    S.lut[1] = __fadd_rn(0.0f, S.ssc[0]);
  }
  consumers_sync();
  for (int k = 1; k < nl; ++k) {
    const float sk = S.ssc[k];
    for (int p = threadIdx.x; p < (1 << k); p += kThreads) {
      const float old = S.lut[p];
      S.lut[p] = __fadd_rn(old, -sk);
      S.lut[p + (1 << k)] = __fadd_rn(old, sk);
    }
    consumers_sync();
  }
  if (n > kLutBits) {
    for (int p = threadIdx.x; p < 16 * 32; p += kThreads) {
      const int pat = p >> 5;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float sj = kLutBits + j < n ? S.ssc[kLutBits + j] : 0.0f;
        v[j] = ((pat >> j) & 1) ? sj : -sj;
      }
      S.quad[p] = make_float4(v[0], v[1], v[2], v[3]);
    }
    consumers_sync();
  }
}

// NW > 0: compiled for exactly NW workers (the common counts), so that the per-element worker checks,
// the sign-byte loads and the division by n fold at compile time; NW = 0: any n up to
// kStageMaxWorkers.  Both compute the same values.  CONTIG: the block walks one contiguous run of
// chunks (run_begin) instead of every gridDim.x-th chunk; the values do not depend on the walk.
template <bool HAS_ERR, int NW, bool CONTIG>
__global__ void __launch_bounds__(kStagedThreads, 3) k_server_staged(const StepArgs A) {
  __shared__ ServerTables S;
  __shared__ volatile int abort_flag;
  __shared__ int redo_squares;  // the chunk's sum of squares is taken again in double
  extern __shared__ __align__(128) unsigned char dyn[];
  const int n = NW > 0 ? NW : A.n;
  const size_t stage_bytes = server_stage_bytes(n);
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + kStages * stage_bytes);
  uint64_t* empty = full + kStages;
  const uint64_t wrow = (uint64_t)A.Wr * 4;  // a multiple of 16: one window offset for all workers
  const uint8_t* wbase = reinterpret_cast<const uint8_t*>(A.wbits);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int st = 0; st < kStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // this block's chunks: every gridDim.x-th from blockIdx.x, or (CONTIG) the run from
  // run_begin(blockIdx.x) up to u_end.  The strided walk reads its first chunk inside each role's
  // branch and its bound and stride from the launch parameters: the same bounds read once before
  // the branch cost the per-tensor kernel 2%, measured.
  const int u_end = CONTIG ? run_begin(A, blockIdx.x + 1) : 0;
  auto in_walk = [&](int u) { return CONTIG ? u < u_end : u < A.n_chunks; };
  // a cursor over this block's (chunk, tile) sequence that keeps the current chunk's descriptor in
  // registers, so that it is read from memory once per chunk rather than at every tile
  struct Cur {
    int u, t, nt;
    Chunk ch;
  };
  auto load = [&](Cur& c) {
    ONEBIT_SKIP_BAD_CHUNKS(c.u, CONTIG ? u_end : A.n_chunks, CONTIG ? 1 : (int)gridDim.x, ONEBIT_K_SERVER);
    if (in_walk(c.u)) {
      c.ch = A.chunks[c.u];
      c.nt = tiles_of(c.ch);
    }
  };
  auto advance = [&](Cur& c) {
    if (++c.t >= c.nt) {
      c.t = 0;
      c.u += CONTIG ? 1 : (int)gridDim.x;
      load(c);
    }
  };

  if (threadIdx.x >= kThreads) {
    // ---------------- producer warp (one elected lane issues the copies)
    if (threadIdx.x != kThreads) return;
    Cur c{CONTIG ? run_begin(A, blockIdx.x) : (int)blockIdx.x, 0, 0, {}};
    load(c);
    int j = 0;
    for (; in_walk(c.u); ++j, advance(c)) {
      const int st = j % kStages;
      if (j >= kStages && !abort_flag && !mbar_wait(&empty[st], (uint32_t)((j / kStages - 1) & 1))) {
        atomicOr(A.status, 2u);
        abort_flag = 1;
      }
      if (abort_flag) break;
      const Chunk& ch = c.ch;
      const int e0 = c.t * kTile;
      const int tlen = min(kTile, ch.len - e0);
      unsigned char* sbase = dyn + (size_t)st * stage_bytes;
      const uint32_t abytes = (uint32_t)(((tlen + 31) / 32) * 32 * 4);  // the padded layout keeps this in bounds
      const uint64_t byte0 = (uint64_t)(ch.off + e0) >> 3;
      const uint32_t nb = (uint32_t)((tlen + 7) / 8);
      // every worker's sign bytes for the tile, widened to the same 16-byte aligned window
      const uint64_t wlo = byte0 & ~(uint64_t)15;
      const uint32_t wlen = (uint32_t)(((byte0 & 15) + nb + 15) & ~(uint64_t)15);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx(&full[st], (HAS_ERR ? abytes : 0u) + (uint32_t)n * wlen + A.stall_tx);
      if (HAS_ERR) bulk_copy_g2s(sbase, A.a + ch.off + e0, abytes, &full[st]);
      for (int i = 0; i < n; ++i)
        bulk_copy_g2s(sbase + (size_t)kTile * 4 + (size_t)i * kRowBytes, wbase + (uint64_t)i * wrow + wlo, wlen,
                      &full[st]);
    }
    if (abort_flag) {
      // drain this block's copies still in flight before the shared memory is released; a second
      // expired wait ends the drain (the copies behind it are as stuck as the first)
      for (int q = j - kStages; q < j; ++q)
        if (q >= 0 && !mbar_wait(&full[q % kStages], (uint32_t)((q / kStages) & 1))) break;
    }
    return;
  }

  // ---------------- consumer warps
  const int lane = threadIdx.x & 31;
  Cur cons{CONTIG ? run_begin(A, blockIdx.x) : (int)blockIdx.x, 0, 0, {}};
  load(cons);
  int k = 0;
  int cur_seg = -1;
  unsigned long long hi = 0, lo = 0;
  while (in_walk(cons.u)) {
    const Chunk ch = cons.ch;
    if (cons.t == 0 && ch.seg != cur_seg) {
      build_server_tables_consumers(S, A, ch.seg);
      cur_seg = ch.seg;
    }
    const int st = k % kStages;
    if (!abort_flag && !mbar_wait(&full[st], (uint32_t)((k / kStages) & 1))) {
      atomicOr(A.status, 2u);
      abort_flag = 1;
    }
    if (!abort_flag) {
      const unsigned char* sbase = dyn + (size_t)st * stage_bytes;
      const float* as = reinterpret_cast<const float*>(sbase);
      const unsigned char* bs = sbase + (size_t)kTile * 4;
      const int e0 = cons.t * kTile;
      const int tlen = min(kTile, ch.len - e0);
      const int boff = (int)(((uint64_t)(ch.off + e0) >> 3) & 15);  // the tile's first byte in each window
      const float Sp = HAS_ERR ? A.sscale_prev[(int64_t)ch.seg * n + ch.shard] : 0.0f;
      // one 8-element group: gl = its index in the tile, cnt = its valid elements
      auto group = [&](const int gl, const int cnt) {
        uint32_t b[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = i < n ? (uint32_t)bs[i * kRowBytes + boff + gl] : 0u;
        float ap[8];
        if (HAS_ERR) {
          const float4 v0 = *reinterpret_cast<const float4*>(as + gl * 8);
          const float4 v1 = *reinterpret_cast<const float4*>(as + gl * 8 + 4);
          ap[0] = v0.x; ap[1] = v0.y; ap[2] = v0.z; ap[3] = v0.w;
          ap[4] = v1.x; ap[5] = v1.y; ap[6] = v1.z; ap[7] = v1.w;
        }
        float sum[8];
        server_sum16(S, n, b, sum);
        for (int i = 16; i < n; ++i) server_add_worker(sum, S.ssc[i], bs[i * kRowBytes + boff + gl]);
        float out[8];
        const uint32_t byte = server_finish<HAS_ERR, NW>(A, sum, ap, Sp, cnt, out, hi, lo);
        const int64_t e = (int64_t)ch.off + e0 + gl * 8;
        store_a(A.a, e, cnt, out);
        reinterpret_cast<uint8_t*>(A.sbits)[e >> 3] = (uint8_t)byte;
      };
      if (tlen == kTile) {
        // a full tile: both groups unguarded in one straight-line block, so that the compiler can
        // interleave their independent work (6-8% faster than the guarded loop, measured)
#pragma unroll
        for (int h = 0; h < kTile / 8 / kThreads; ++h) group(threadIdx.x + h * kThreads, 8);
      } else {
        for (int h = 0; h < kTile / 8 / kThreads; ++h) {
          const int gl = threadIdx.x + h * kThreads;
          if (gl * 8 < tlen) group(gl, tlen - gl * 8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with stage st
    }
    ++k;
    const bool last_tile = cons.t == cons.nt - 1;
    const int u_done = cons.u;
    advance(cons);
    if (last_tile) {  // chunk total among the consumers (fixed order)
      consumers_total(sq_of(hi, lo), S.red, &redo_squares, &abort_flag);
      if (redo_squares && threadIdx.x < 32) {  // outside the exact range: warp 0 sums the chunk again in double
        const Chunk cd = A.chunks[u_done];  // reloaded: keeping the descriptor live costs registers
        const double r = warp_sum(squares_fp64(A.a + cd.off, cd.len, threadIdx.x, 32));
        if (threadIdx.x == 0) S.red[kConsumerWarps] = r;
      }
      if (threadIdx.x == 0 && !abort_flag) A.spart[u_done] = S.red[kConsumerWarps];
      hi = lo = 0;
    }
  }
}

// ------------------------------------------------------------------------------------------------
// K3: broadcast unpack + preconditioned update  x = x - lr * (m / den),  m = S_kj * sign(a).
// SPANS: walk the worker-side chunks instead of the server-side ones.  Plans whose shards are much
// shorter than a chunk (short scale blocks) have worker chunks that hold several whole shards; each
// 8-element group then takes the scale of its own shard, and the units stay long.

template <bool VEC, bool SPANS = false>
__global__ void __launch_bounds__(kThreads) k_update(const StepArgs A) {
  const float lr = A.lr;
  for (int u = blockIdx.x; u < (SPANS ? A.n_wchunks : A.n_chunks); u += gridDim.x) {
    const Chunk ch = (SPANS ? A.wchunks : A.chunks)[u];
    ONEBIT_CHECK_UNIT(chunk_ok(A, ch) && ch.per >= 0 && (ch.per == 0 || ch.shard + (ch.len - 1) / ch.per < A.n),
                      A.status, ONEBIT_K_UPDATE)
    const float S = A.sscale_cur[(int64_t)ch.seg * A.n + ch.shard];
    // SPANS: a group's shard is the chunk's first plus its offset / the shard length
    const float* __restrict__ Sseg = A.sscale_cur + (int64_t)ch.seg * A.n + ch.shard;
    auto scale_of = [&](int gi) { return ch.per ? Sseg[(uint32_t)(gi * 8) / (uint32_t)ch.per] : S; };
    float* __restrict__ x = A.pptr[ch.seg] + ch.start;
    const float* __restrict__ den = A.v + ch.off;
    const uint8_t* __restrict__ sb = reinterpret_cast<const uint8_t*>(A.sbits) + (ch.off >> 3);
    struct In {
      float x[8], d[8];
      uint32_t b;
      float S;
    };
    auto load = [&](In& r, int gi) {
      const int64_t e = (int64_t)gi * 8;
      if (VEC) ld8_state(x + e, r.x);
      else
#pragma unroll
        for (int q = 0; q < 8; ++q) r.x[q] = x[e + q];
      ld8_stream(den + e, r.d);
      r.b = sb[gi];
      if (SPANS) r.S = scale_of(gi);
    };
    auto work = [&](In& r, int gi) {
      const int64_t e = (int64_t)gi * 8;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float Sg = SPANS ? r.S : S;
        const float mq = ((r.b >> q) & 1u) ? Sg : -Sg;
        r.x[q] = __fsub_rn(r.x[q], __fmul_rn(lr, __fdiv_rn(mq, r.d[q])));
      }
      if (VEC) st8(x + e, r.x);
      else
#pragma unroll
        for (int q = 0; q < 8; ++q) x[e + q] = r.x[q];
    };
    const int ng = ch.len >> 3;
    int gi = threadIdx.x;
    for (; gi + kThreads < ng; gi += 2 * kThreads) {
      In r0, r1;
      load(r0, gi);
      load(r1, gi + kThreads);
      work(r0, gi);
      work(r1, gi + kThreads);
    }
    if (gi < ng) {
      In r0;
      load(r0, gi);
      work(r0, gi);
    }
    const int rem = ch.len & 7;
    if (rem && threadIdx.x == (ng % kThreads)) {
      const int64_t e0 = (int64_t)ng * 8;
      const float St = SPANS ? scale_of(ng) : S;
      for (int q = 0; q < rem; ++q) {
        const float mq = ((sb[ng] >> q) & 1u) ? St : -St;
        x[e0 + q] = __fsub_rn(x[e0 + q], __fmul_rn(lr, __fdiv_rn(mq, den[e0 + q])));
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// Gradient-compression baseline: every worker runs Adam on the broadcast g_hat = S * sign(a).

template <bool BC, bool VEC>
__global__ void __launch_bounds__(kThreads) k_ec_adam_update(const StepArgs A) {
  for (int u = blockIdx.x; u < A.n_chunks; u += gridDim.x) {
    const Chunk ch = A.chunks[u];
    ONEBIT_CHECK_UNIT(chunk_ok(A, ch), A.status, ONEBIT_K_EC_UPDATE)
    const float S = A.sscale_cur[(int64_t)ch.seg * A.n + ch.shard];
    float* __restrict__ x = A.pptr[ch.seg] + ch.start;
    float* __restrict__ m = A.m + ch.off;
    float* __restrict__ v = A.v + ch.off;
    const uint8_t* __restrict__ sb = reinterpret_cast<const uint8_t*>(A.sbits) + (ch.off >> 3);
    const int ng = (ch.len + 7) >> 3;
    for (int gi = threadIdx.x; gi < ng; gi += kThreads) {
      const int cnt = min(8, ch.len - gi * 8);
      const int64_t e = (int64_t)gi * 8;
      const bool vec = VEC && cnt == 8;
      float mv[8], vv[8], xv[8];
      if (cnt == 8) {
        ld8_state(m + e, mv);
        ld8_state(v + e, vv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          mv[q] = q < cnt ? m[e + q] : 0.0f;
          vv[q] = q < cnt ? v[e + q] : 0.0f;
        }
      }
      if (vec) {
        ld8_state(x + e, xv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[q] = q < cnt ? x[e + q] : 0.0f;
      }
      const uint32_t byte = sb[gi];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float gh = ((byte >> q) & 1u) ? S : -S;
        mv[q] = momentum(A.b1, A.omb1, mv[q], gh);
        vv[q] = __fadd_rn(__fmul_rn(A.b2, vv[q]), __fmul_rn(A.omb2, __fmul_rn(gh, gh)));
        const float mh = BC ? __fdiv_rn(mv[q], A.bc1) : mv[q];
        const float vh = BC ? __fdiv_rn(vv[q], A.bc2) : vv[q];
        xv[q] = __fsub_rn(xv[q], __fmul_rn(A.lr, __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), A.eps))));
      }
      if (cnt == 8) {
        st8(m + e, mv);
        st8(v + e, vv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < cnt) {
            m[e + q] = mv[q];
            v[e + q] = vv[q];
          }
      }
      if (vec) {
        st8(x + e, xv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < cnt) x[e + q] = xv[q];
      }
    }
  }
}

// ------------------------------------------------------------------------------------------------
// K0: warm-up.  Mean of the n worker gradients (summed in worker order), then one Adam step.
// The gradients are fetched in batches whose loads are all issued before the batch is added in order,
// so one memory latency covers a whole batch.  Large batches (16 workers for 16-bit, 8 for fp32
// gradients) hold the kernel to 128 registers, two CTAs per SM; for n <= 4 16-bit gradients a batch
// of 4 needs far fewer registers and the kernel runs three CTAs per SM.

template <typename GT> struct RawGrad;  // one 8-element gradient group as loaded
template <> struct RawGrad<float> {
  float v[8];
  __device__ __forceinline__ void load(const float* p) { ld8_stream(p, v); }
  __device__ __forceinline__ float get(int q) const { return v[q]; }
};
template <> struct RawGrad<__half> {
  uint4 u;
  __device__ __forceinline__ void load(const __half* p) { u = ld16_stream(p); }
  __device__ __forceinline__ float get(int q) const {
    const uint32_t w = q < 2 ? u.x : q < 4 ? u.y : q < 6 ? u.z : u.w;
    return __half2float(__ushort_as_half((unsigned short)((q & 1) ? (w >> 16) : (w & 0xffffu))));
  }
};
template <> struct RawGrad<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { u = ld16_stream(p); }
  __device__ __forceinline__ float get(int q) const {
    const uint32_t w = q < 2 ? u.x : q < 4 ? u.y : q < 6 ? u.z : u.w;
    return __uint_as_float((q & 1) ? (w & 0xffff0000u) : (w << 16));
  }
};

// With MON the kernel also writes each chunk's exact sum of the new v^2 to A.spart (the "fused
// variance norm" monitor; k_variance_norm reduces it).
template <typename GT, bool BC, bool VEC, bool MON, bool SMALL>
__global__ void __launch_bounds__(kThreads, SMALL ? 3 : 2) k_warmup(const StepArgs A) {
  constexpr int B = SMALL ? 4 : (sizeof(GT) == 4 ? 8 : 16);
  __shared__ const GT* gsm[kMaxWorkers];
  __shared__ double red[kThreads / 32 + 2];
  for (int u = blockIdx.x; u < A.n_chunks; u += gridDim.x) {
    unsigned long long vhi = 0, vlo = 0;
    const Chunk ch = A.chunks[u];
    ONEBIT_CHECK_UNIT(chunk_ok(A, ch), A.status, ONEBIT_K_WARMUP)
    __syncthreads();
    for (int i = threadIdx.x; i < A.n; i += kThreads)
      gsm[i] = static_cast<const GT*>(A.gptr[(int64_t)i * A.T + ch.seg]) + ch.start;
    __syncthreads();
    float* __restrict__ x = A.pptr[ch.seg] + ch.start;
    float* __restrict__ m = A.m + ch.off;
    float* __restrict__ v = A.v + ch.off;
    const int ng = (ch.len + 7) >> 3;
    for (int gi = threadIdx.x; gi < ng; gi += kThreads) {
      const int cnt = min(8, ch.len - gi * 8);
      const int64_t e = (int64_t)gi * 8;
      const bool vec = VEC && cnt == 8;
      float mv[8], vv[8], xv[8];
      if (cnt == 8) {
        ld8_state(m + e, mv);
        ld8_state(v + e, vv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          mv[q] = q < cnt ? m[e + q] : 0.0f;
          vv[q] = q < cnt ? v[e + q] : 0.0f;
        }
      }
      if (vec) {
        ld8_state(x + e, xv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) xv[q] = q < cnt ? x[e + q] : 0.0f;
      }
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
      for (int i0 = 0; i0 < A.n; i0 += B) {
        if (vec) {
          RawGrad<GT> r[B];
#pragma unroll
          for (int j = 0; j < B; ++j)
            if (i0 + j < A.n) r[j].load(gsm[i0 + j] + e);
#pragma unroll
          for (int j = 0; j < B; ++j)
            if (i0 + j < A.n)
#pragma unroll
              for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], r[j].get(q));
        } else {
          for (int j = 0; j < B && i0 + j < A.n; ++j) {
            const GT* gp = gsm[i0 + j] + e;
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], q < cnt ? Grad<GT>::load1(gp + q) : 0.0f);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float gbar = A.pow2 ? __fmul_rn(acc[q], A.inv_n) : __fdiv_rn(acc[q], A.nf);
        mv[q] = momentum(A.b1, A.omb1, mv[q], gbar);
        vv[q] = __fadd_rn(__fmul_rn(A.b2, vv[q]), __fmul_rn(A.omb2, __fmul_rn(gbar, gbar)));
        const float mh = BC ? __fdiv_rn(mv[q], A.bc1) : mv[q];
        const float vh = BC ? __fdiv_rn(vv[q], A.bc2) : vv[q];
        xv[q] = __fsub_rn(xv[q], __fmul_rn(A.lr, __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), A.eps))));
      }
      if (MON) {
#pragma unroll
        for (int q = 0; q < 8; q += 2) add_square2(vhi, vlo, q < cnt ? vv[q] : 0.0f, q + 1 < cnt ? vv[q + 1] : 0.0f);
      }
      if (cnt == 8) {
        st8(m + e, mv);
        st8(v + e, vv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < cnt) {
            m[e + q] = mv[q];
            v[e + q] = vv[q];
          }
      }
      if (vec) {
        st8(x + e, xv);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < cnt) x[e + q] = xv[q];
      }
    }
    if (MON) {
      const double tot = unit_squares<kThreads>(vhi, vlo, v, ch.len, red);
      if (threadIdx.x == 0) A.spart[u] = tot;
    }
  }
}

// K0, staged variant: 16-bit gradients, kWarmStagedMin <= n <= kWarmStagedMax, every pointer
// aligned.  Per-thread register batches cannot keep enough bytes in flight for 16 gradient streams
// read 16 bytes at a time, so a producer warp streams each tile of the n gradient rows and of m, v
// and x into shared memory with bulk copies (two stages), and the consumer warps add the gradients
// in worker order and run the same fp32 Adam arithmetic as k_warmup, writing m, v and x straight
// back.  A tile's last partial group (a tensor's ragged end) is read with plain loads.  Waits are
// bounded exactly as in the staged server kernel.
constexpr int kWTile = 2048;   // elements per tile: one 8-element group per consumer thread
constexpr int kWStages = 2;
constexpr int kWarmStagedMin = 8;
constexpr int kWarmStagedMax = 20;  // two stages of 2048 * (2n + 12) bytes fit the 227 KB per CTA
__host__ __device__ constexpr size_t warmup_stage_bytes(int n) { return (size_t)kWTile * (2 * n + 12); }
__host__ __device__ constexpr size_t warmup_dyn_smem(int n) { return kWStages * warmup_stage_bytes(n) + 2 * kWStages * 8; }

template <typename GT, bool BC, bool MON>
__global__ void __launch_bounds__(kStagedThreads) k_warmup_staged(const StepArgs A) {
  __shared__ double red[kConsumerWarps + 2];
  __shared__ volatile int abort_flag;
  __shared__ int redo_squares;  // the chunk's sum of squares is taken again in double
  extern __shared__ __align__(128) unsigned char dyn[];
  const int n = A.n;
  const size_t stage_bytes = warmup_stage_bytes(n);
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + kWStages * stage_bytes);
  uint64_t* empty = full + kWStages;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int st = 0; st < kWStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  auto advance = [&](TileCursor& c) {
    if (++c.t >= (A.chunks[c.u].len + kWTile - 1) / kWTile) {
      c.t = 0;
      c.u += gridDim.x;
      ONEBIT_SKIP_BAD_CHUNKS(c.u, A.n_chunks, (int)gridDim.x, ONEBIT_K_WARMUP);
    }
  };
  const size_t mofs = (size_t)n * kWTile * 2;  // stage layout: n gradient rows, then m, v, x

  if (threadIdx.x >= kThreads) {
    // ---------------- producer warp (one elected lane issues the copies)
    if (threadIdx.x != kThreads) return;
    TileCursor c{(int)blockIdx.x, 0};
    ONEBIT_SKIP_BAD_CHUNKS(c.u, A.n_chunks, (int)gridDim.x, ONEBIT_K_WARMUP);
    int j = 0;
    for (; c.u < A.n_chunks; ++j, advance(c)) {
      const int st = j % kWStages;
      if (j >= kWStages && !abort_flag && !mbar_wait(&empty[st], (uint32_t)((j / kWStages - 1) & 1))) {
        atomicOr(A.status, 2u);
        abort_flag = 1;
      }
      if (abort_flag) break;
      const Chunk ch = A.chunks[c.u];
      const int e0 = c.t * kWTile;
      const int tv = min(kWTile, ch.len - e0) & ~7;  // whole groups: every copy a multiple of 16 bytes
      unsigned char* sb = dyn + (size_t)st * stage_bytes;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_expect_tx(&full[st], (uint32_t)tv * (uint32_t)(2 * n + 12) + A.stall_tx);
      if (tv > 0) {
        for (int i = 0; i < n; ++i)
          bulk_copy_g2s(sb + (size_t)i * kWTile * 2,
                        static_cast<const GT*>(A.gptr[(int64_t)i * A.T + ch.seg]) + ch.start + e0, (uint32_t)tv * 2,
                        &full[st]);
        bulk_copy_g2s(sb + mofs, A.m + ch.off + e0, (uint32_t)tv * 4, &full[st]);
        bulk_copy_g2s(sb + mofs + kWTile * 4, A.v + ch.off + e0, (uint32_t)tv * 4, &full[st]);
        bulk_copy_g2s(sb + mofs + kWTile * 8, A.pptr[ch.seg] + ch.start + e0, (uint32_t)tv * 4, &full[st]);
      }
    }
    if (abort_flag) {
      for (int q = j - kWStages; q < j; ++q)
        if (q >= 0 && !mbar_wait(&full[q % kWStages], (uint32_t)((q / kWStages) & 1))) break;
    }
    return;
  }

  // ---------------- consumer warps: thread t owns elements [8t, 8t+8) of every tile
  const int lane = threadIdx.x & 31;
  TileCursor cons{(int)blockIdx.x, 0};
  ONEBIT_SKIP_BAD_CHUNKS(cons.u, A.n_chunks, (int)gridDim.x, ONEBIT_K_WARMUP);
  int k = 0;
  unsigned long long vhi = 0, vlo = 0;
  while (cons.u < A.n_chunks) {
    const Chunk ch = A.chunks[cons.u];
    const int st = k % kWStages;
    if (!abort_flag && !mbar_wait(&full[st], (uint32_t)((k / kWStages) & 1))) {
      atomicOr(A.status, 2u);
      abort_flag = 1;
    }
    if (!abort_flag) {
      const unsigned char* sb = dyn + (size_t)st * stage_bytes;
      const int e0 = cons.t * kWTile;
      const int tlen = min(kWTile, ch.len - e0);
      const int eg = threadIdx.x * 8;
      if (eg < tlen) {
        const int cnt = min(8, tlen - eg);
        const int64_t ge = (int64_t)e0 + eg;  // element within the chunk
        float* m = A.m + ch.off + ge;
        float* v = A.v + ch.off + ge;
        float* x = A.pptr[ch.seg] + ch.start + ge;
        float mv[8], vv[8], xv[8], acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        if (eg + 8 <= (tlen & ~7)) {  // the whole group is in the stage
          const float4* ms = reinterpret_cast<const float4*>(sb + mofs) + eg / 4;
          const float4* vs = reinterpret_cast<const float4*>(sb + mofs + kWTile * 4) + eg / 4;
          const float4* xs = reinterpret_cast<const float4*>(sb + mofs + kWTile * 8) + eg / 4;
          const float4 m0 = ms[0], m1 = ms[1], v0 = vs[0], v1 = vs[1], x0 = xs[0], x1 = xs[1];
          mv[0] = m0.x; mv[1] = m0.y; mv[2] = m0.z; mv[3] = m0.w; mv[4] = m1.x; mv[5] = m1.y; mv[6] = m1.z; mv[7] = m1.w;
          vv[0] = v0.x; vv[1] = v0.y; vv[2] = v0.z; vv[3] = v0.w; vv[4] = v1.x; vv[5] = v1.y; vv[6] = v1.z; vv[7] = v1.w;
          xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w; xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
          for (int i = 0; i < n; ++i) {
            RawGrad<GT> r;
            r.u = *reinterpret_cast<const uint4*>(sb + (size_t)i * kWTile * 2 + (size_t)eg * 2);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], r.get(q));
          }
        } else {  // a tensor's ragged end: plain loads
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            mv[q] = q < cnt ? m[q] : 0.0f;
            vv[q] = q < cnt ? v[q] : 0.0f;
            xv[q] = q < cnt ? x[q] : 0.0f;
          }
          for (int i = 0; i < n; ++i) {
            const GT* gp = static_cast<const GT*>(A.gptr[(int64_t)i * A.T + ch.seg]) + ch.start + ge;
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = __fadd_rn(acc[q], q < cnt ? Grad<GT>::load1(gp + q) : 0.0f);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float gbar = A.pow2 ? __fmul_rn(acc[q], A.inv_n) : __fdiv_rn(acc[q], A.nf);
          mv[q] = momentum(A.b1, A.omb1, mv[q], gbar);
          vv[q] = __fadd_rn(__fmul_rn(A.b2, vv[q]), __fmul_rn(A.omb2, __fmul_rn(gbar, gbar)));
          const float mh = BC ? __fdiv_rn(mv[q], A.bc1) : mv[q];
          const float vh = BC ? __fdiv_rn(vv[q], A.bc2) : vv[q];
          xv[q] = __fsub_rn(xv[q], __fmul_rn(A.lr, __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), A.eps))));
        }
        if (MON) {
#pragma unroll
          for (int q = 0; q < 8; q += 2)
            add_square2(vhi, vlo, q < cnt ? vv[q] : 0.0f, q + 1 < cnt ? vv[q + 1] : 0.0f);
        }
        if (cnt == 8) {
          st8(m, mv);
          st8(v, vv);
          st8(x, xv);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < cnt) {
              m[q] = mv[q];
              v[q] = vv[q];
              x[q] = xv[q];
            }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    ++k;
    const bool last_tile = cons.t == (ch.len + kWTile - 1) / kWTile - 1;
    const int u_done = cons.u;
    advance(cons);
    if (MON && last_tile) {  // chunk total of v^2 among the consumers (fixed order)
      consumers_total(sq_of(vhi, vlo), red, &redo_squares, &abort_flag);
      if (redo_squares && threadIdx.x < 32) {  // outside the exact range: warp 0 sums the chunk again in double
        const Chunk cd = A.chunks[u_done];
        const double r = warp_sum(squares_fp64(A.v + cd.off, cd.len, threadIdx.x, 32));
        if (threadIdx.x == 0) red[kConsumerWarps] = r;
      }
      if (threadIdx.x == 0 && !abort_flag) A.spart[u_done] = red[kConsumerWarps];
      vhi = vlo = 0;
    }
  }
}

// ||v||_2 after a monitored warm-up step: one CTA, fixed-order sum of the chunk partials.
static __global__ void __launch_bounds__(kScaleThreads) k_variance_norm(const double* part, int n_chunks, double* out) {
  __shared__ double red[kScaleThreads / 32];
  double acc = 0.0;
  for (int c = threadIdx.x; c < n_chunks; c += kScaleThreads) acc += __ldcg(part + c);
  const double tot = block_sum<kScaleThreads>(acc, red);
  if (threadIdx.x == 0) *out = sqrt(tot);
}

// ------------------------------------------------------------------------------------------------
// KF: freeze  den = sqrt(v) + eps  (v / bc2 first with bias correction), in place over Dp.

template <bool BC>
__global__ void __launch_bounds__(kThreads) k_freeze(float* v, int64_t n_groups, float bc2, float eps) {
  for (int64_t gi = blockIdx.x * (int64_t)kThreads + threadIdx.x; gi < n_groups;
       gi += (int64_t)gridDim.x * kThreads) {
    float r[8];
    ld8_state(v + gi * 8, r);
#pragma unroll
    for (int q = 0; q < 8; ++q) r[q] = __fadd_rn(__fsqrt_rn(BC ? __fdiv_rn(r[q], bc2) : r[q]), eps);
    st8(v + gi * 8, r);
  }
}

// ------------------------------------------------------------------------------------------------
// Exchange copies of the multi-GPU form: word ranges between this rank's state and the caller's
// exchange buffers (the messages each peer's servers need, and this rank's share of the broadcast).
// Regions: 0 worker sign rows, 1 current worker scales, 2 server sign words, 3 current server scales,
// 4 the caller's exchange buffer.  Offsets and lengths are in 32-bit words (scales are copied bit for
// bit).

struct XRange {
  int64_t src, dst;  // word offsets within the source and destination regions
  int32_t len;       // words, <= kXPiece
  int16_t sreg, dreg;
};
constexpr int kXPiece = 8192;  // longer ranges are cut into pieces of this many words

struct XArgs {
  const XRange* r;
  int32_t n;
  uint32_t* base[5];
#ifdef ONEBIT_CHECKS
  int64_t words[5];       // each region's extent in words
  unsigned int* status;
#endif
};

static __global__ void __launch_bounds__(kThreads) k_exchange_copy(const XArgs X) {
  for (int q = blockIdx.x; q < X.n; q += gridDim.x) {
    const XRange r = X.r[q];
    ONEBIT_CHECK_UNIT(r.len >= 0 && r.len <= kXPiece && r.sreg >= 0 && r.sreg < 5 && r.dreg >= 0 && r.dreg < 5 &&
                          r.src >= 0 && r.src + r.len <= X.words[r.sreg] && r.dst >= 0 &&
                          r.dst + r.len <= X.words[r.dreg],
                      X.status, ONEBIT_K_EXCHANGE)
    const uint32_t* s = X.base[r.sreg] + r.src;
    uint32_t* d = X.base[r.dreg] + r.dst;
    for (int e = threadIdx.x; e < r.len; e += kThreads) d[e] = s[e];
  }
}

// ------------------------------------------------------------------------------------------------
// Export / import between the padded state layout and the caller's unpadded fp32 layout.

enum ExportKind : int {
  kExportCopy = 0,      // dst = src                        (m dense, v/den)
  kExportSignedErr = 1, // dst = err(src, scale[seg...])    (worker / server error)
  kExportBits = 2,      // dst = bit ? S : -S               (m from the broadcast)
  kExportZero = 3,      // dst = 0
  kImportCopy = 4       // padded dst = unpadded src
};

struct ExportArgs {
  const Chunk* chunks;
  int32_t n_chunks;
  int32_t kind;
  int32_t scale_stride;  // index of the scale: seg*scale_seg_mul + shard*scale_shard_mul
  int32_t scale_seg_mul;
  int32_t scale_shard_mul;
  int32_t pad_;
  const float* src;      // padded source (or unpadded source for import)
  const uint32_t* bits;  // sign words for kExportBits
  const float* scales;
  float* dst;
#ifdef ONEBIT_CHECKS
  int64_t Dp, D;          // padded and unpadded elements of the state and of the caller's buffer
  int64_t n_scales;       // entries of `scales`
  unsigned int* status;
#endif
};

static __global__ void __launch_bounds__(kThreads) k_export(const ExportArgs X) {
  for (int u = blockIdx.x; u < X.n_chunks; u += gridDim.x) {
    const Chunk ch = X.chunks[u];
    ONEBIT_CHECK_UNIT(ch.len >= 0 && ch.off >= 0 && ch.off + ch.len <= X.Dp && ch.uoff >= 0 &&
                          ch.uoff + ch.len <= X.D &&
                          (!X.scales || ((int64_t)ch.seg * X.scale_seg_mul + (int64_t)ch.shard * X.scale_shard_mul >= 0 &&
                                         (int64_t)ch.seg * X.scale_seg_mul + (int64_t)ch.shard * X.scale_shard_mul <
                                             X.n_scales)),
                      X.status, ONEBIT_K_EXPORT)
    const float s = X.scales ? X.scales[(int64_t)ch.seg * X.scale_seg_mul + (int64_t)ch.shard * X.scale_shard_mul]
                             : 0.0f;
    for (int e = threadIdx.x; e < ch.len; e += kThreads) {
      const int64_t p = ch.off + e, q = ch.uoff + e;
      switch (X.kind) {
        case kExportCopy: X.dst[q] = X.src[p]; break;
        case kExportSignedErr: X.dst[q] = error_of(X.src[p], s); break;
        case kExportBits: X.dst[q] = ((X.bits[p >> 5] >> (p & 31)) & 1u) ? s : -s; break;
        case kExportZero: X.dst[q] = 0.0f; break;
        case kImportCopy: X.dst[p] = X.src[q]; break;
        default: break;
      }
    }
  }
}

}  // namespace onebit
