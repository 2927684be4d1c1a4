// onebit_noalloc.cu -- worker compression of one vector with no device allocation.
//
// Some callers cannot allocate device memory at the point where they need this operation: code
// running under a framework whose caching allocator owns every device byte (a raw cudaMalloc would
// bypass its accounting and can synchronise the whole device), latency-critical loops where that
// implicit synchronisation is not acceptable, or plug-ins that are given buffers but no right to
// allocate.  onebit_worker_compress_noalloc() serves them: the caller passes only inputs and outputs,
// and the scratch the computation needs (per-chunk sum-of-squares partials and the scale) lives in a
// file-scope __device__ array that every GPU loading this library holds until the process exits.
//
// It is the worker kernel of the compression step run for one vector (65536-element chunks): the
// same per-element fp32 operation order and the same exact-square norm, so its sign bits equal
// those of onebit_adam_compress_step() for the same vector, and its scale (hence its error) agrees to
// within one fp32 rounding of the scale (the handle may group the norm's partial sums into shorter
// chunks).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/onebit_adam.h"
#include "onebit_kernels.cuh"

namespace onebit {
namespace {

constexpr int kNoAllocParts = ONEBIT_NOALLOC_MAX_LEN / kChunk;  // 4096 partials
constexpr int kNoAllocMaxDevices = 64;

// [0, kNoAllocParts): per-chunk partials; [kNoAllocParts]: the scale.  Every slot a call reads is
// written earlier in the same call, so nothing has to be cleared between calls; calls that overlap
// on the GPU (different streams, no ordering) race on this array.
static __device__ __align__(256) double g_scratch[kNoAllocParts + 32];

// Pass 1: c = (b1*m + (1-b1)*g) + err_in, its sign bits, and each chunk's sum of c^2.
// c is written to the error output and turned into the error by pass 3.
template <typename GT, bool HAS_ERR, bool VEC>
__global__ void __launch_bounds__(kThreads) k_vec_worker(const float* __restrict__ m, const GT* __restrict__ g,
                                                         const float* err_in, float b1, float omb1, int64_t len,
                                                         int n_chunks, uint8_t* __restrict__ bits, float* c,
                                                         double* part) {
  __shared__ double red[kThreads / 32 + 2];
  for (int ci = blockIdx.x; ci < n_chunks; ci += gridDim.x) {
    const int64_t base = (int64_t)ci * kChunk;
    const int clen = (int)(len - base < kChunk ? len - base : kChunk);
    const float* mc = m + base;
    const GT* gc = g + base;
    const float* ec = HAS_ERR ? err_in + base : nullptr;
    float* cc = c + base;
    uint8_t* bc = bits + (base >> 3);
    struct In {
      float g[8], e[8], m[8];
    };
    auto load = [&](In& r, int gi) {
      const int64_t e = (int64_t)gi * 8;
      if (VEC) {
        Grad<GT>::load8(gc + e, r.g);
        ld8_stream(mc + e, r.m);
        if (HAS_ERR) ld8_state(ec + e, r.e);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          r.g[q] = Grad<GT>::load1(gc + e + q);
          r.m[q] = mc[e + q];
          if (HAS_ERR) r.e[q] = ec[e + q];
        }
      }
    };
    unsigned long long hi = 0, lo = 0;
    auto work = [&](const In& r, int gi) {
      float out[8];
      uint32_t byte = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float mi = momentum(b1, omb1, r.m[q], r.g[q]);
        const float cq = __fadd_rn(mi, HAS_ERR ? r.e[q] : 0.0f);
        out[q] = cq;
        byte |= (cq >= 0.0f ? 1u : 0u) << q;
      }
#pragma unroll
      for (int q = 0; q < 8; q += 2) add_square2(hi, lo, out[q], out[q + 1]);
      if (VEC) {
        st8(cc + (int64_t)gi * 8, out);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) cc[(int64_t)gi * 8 + q] = out[q];
      }
      bc[gi] = (uint8_t)byte;
    };
    const int ng = clen >> 3;
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
    const int rem = clen & 7;
    if (rem && threadIdx.x == (ng % kThreads)) {
      const int64_t e0 = (int64_t)ng * 8;
      uint32_t byte = 0;
      for (int q = 0; q < rem; ++q) {
        const int64_t e = e0 + q;
        const float mi = momentum(b1, omb1, mc[e], Grad<GT>::load1(gc + e));
        const float cq = __fadd_rn(mi, HAS_ERR ? ec[e] : 0.0f);
        cc[e] = cq;
        byte |= (cq >= 0.0f ? 1u : 0u) << q;
        add_square2(hi, lo, cq, 0.0f);
      }
      bc[ng] = (uint8_t)byte;
    }
    if (base + clen == len && threadIdx.x == 0) {
      // the caller's last sign word may hold anything: zero its bytes past the vector's end
      const int64_t used = (len + 7) >> 3, words = (len + 31) >> 5;
      for (int64_t b = used; b < words * 4; ++b) bits[b] = 0;
    }
    const double tot = unit_squares<kThreads>(hi, lo, cc, clen, red);
    if (threadIdx.x == 0) part[ci] = tot;
  }
}

// Pass 2: one CTA sums the partials in a fixed order (as the handle's scale kernel does).
__global__ void __launch_bounds__(kScaleThreads) k_vec_scale(double* part, int n_chunks, int64_t len,
                                                             float* scale_out) {
  __shared__ double red[kScaleThreads / 32];
  double acc = 0.0;
  for (int c = threadIdx.x; c < n_chunks; c += kScaleThreads) acc += __ldcg(part + c);
  const double tot = block_sum<kScaleThreads>(acc, red);
  if (threadIdx.x == 0) {
    const float s = __double2float_rn(sqrt(tot / (double)len));
    part[kNoAllocParts] = (double)s;
    *scale_out = s;
  }
}

// Pass 3: error = c - scale*sign(c), in place.
__global__ void __launch_bounds__(kThreads) k_vec_error(float* c, int64_t len, const double* part) {
  const float s = (float)__ldcg(part + kNoAllocParts);
  for (int64_t e = blockIdx.x * (int64_t)kThreads + threadIdx.x; e < len; e += (int64_t)gridDim.x * kThreads)
    c[e] = error_of(c[e], s);
}

// Device address of g_scratch for each device, looked up on that device's first call.
std::mutex g_mu;
void* g_addr[kNoAllocMaxDevices] = {};

cudaError_t scratch_for_current_device(double** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = static_cast<double*>(g_addr[dev]);
  return cudaSuccess;
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename GT>
cudaError_t launch_vec(const float* m, const void* grad, const float* err_in, float b1, int64_t len, uint32_t* bits,
                       float* scale_out, float* err_out, double* part, cudaStream_t st) {
  const GT* g = static_cast<const GT*>(grad);
  const int n_chunks = (int)((len + kChunk - 1) / kChunk);
  const float omb1 = 1.0f - b1;
  const bool vec = al(m, 32) && al(err_out, 32) && (!err_in || al(err_in, 32)) && al(g, sizeof(GT) == 4 ? 32 : 16);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid1 = n_chunks < sms * 4 ? n_chunks : sms * 4;
  uint8_t* b8 = reinterpret_cast<uint8_t*>(bits);
  if (err_in) {
    if (vec) k_vec_worker<GT, true, true><<<grid1, kThreads, 0, st>>>(m, g, err_in, b1, omb1, len, n_chunks, b8, err_out, part);
    else k_vec_worker<GT, true, false><<<grid1, kThreads, 0, st>>>(m, g, err_in, b1, omb1, len, n_chunks, b8, err_out, part);
  } else {
    if (vec) k_vec_worker<GT, false, true><<<grid1, kThreads, 0, st>>>(m, g, nullptr, b1, omb1, len, n_chunks, b8, err_out, part);
    else k_vec_worker<GT, false, false><<<grid1, kThreads, 0, st>>>(m, g, nullptr, b1, omb1, len, n_chunks, b8, err_out, part);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_vec_scale<<<1, kScaleThreads, 0, st>>>(part, n_chunks, len, scale_out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int64_t blocks = (len + kThreads - 1) / kThreads;
  const int grid3 = (int)(blocks < (int64_t)sms * 8 ? blocks : (int64_t)sms * 8);
  k_vec_error<<<grid3, kThreads, 0, st>>>(err_out, len, part);
  return cudaGetLastError();
}

}  // namespace
}  // namespace onebit

extern "C" onebit_status_t onebit_worker_compress_noalloc(const float* m, const void* grad, int32_t grad_dtype,
                                                          const float* err_in, float beta1, int64_t len,
                                                          uint32_t* bits_out, float* scale_out, float* err_out,
                                                          onebit_stream_t stream) {
  using namespace onebit;
  if (!m || !grad || !bits_out || !scale_out || !err_out) return ONEBIT_ERR_INVALID_ARG;
  if (len < 1 || len > ONEBIT_NOALLOC_MAX_LEN) return ONEBIT_ERR_INVALID_ARG;
  if (grad_dtype < ONEBIT_F32 || grad_dtype > ONEBIT_BF16) return ONEBIT_ERR_INVALID_ARG;
  if (!(beta1 >= 0.0f && beta1 < 1.0f)) return ONEBIT_ERR_INVALID_ARG;
  {
    // Every output must be disjoint from every input and from the other outputs (the kernels read
    // the inputs through the read-only cache while the outputs are written), except that err_in may
    // be exactly err_out (updated in place: each element is read before it is written).
    struct Span {
      const char* p;
      int64_t bytes;
    };
    auto span = [](const void* q, int64_t bytes) { return Span{static_cast<const char*>(q), q ? bytes : 0}; };
    auto overlap = [](Span a, Span b) { return a.bytes > 0 && b.bytes > 0 && a.p < b.p + b.bytes && b.p < a.p + a.bytes; };
    const int64_t gb = grad_dtype == ONEBIT_F32 ? 4 : 2;
    const Span in_m = span(m, len * 4), in_g = span(grad, len * gb);
    const Span in_e = span(err_in == err_out ? nullptr : err_in, len * 4);
    const Span out_b = span(bits_out, ((len + 31) / 32) * 4), out_s = span(scale_out, 4), out_e = span(err_out, len * 4);
    for (const Span o : {out_b, out_s, out_e})
      for (const Span i : {in_m, in_g, in_e})
        if (overlap(o, i)) return ONEBIT_ERR_INVALID_ARG;
    if (overlap(out_b, out_s) || overlap(out_b, out_e) || overlap(out_s, out_e)) return ONEBIT_ERR_INVALID_ARG;
  }
  double* part = nullptr;
  if (scratch_for_current_device(&part) != cudaSuccess) {
    cudaGetLastError();
    return ONEBIT_ERR_CUDA;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (grad_dtype) {
    case ONEBIT_F32: e = launch_vec<float>(m, grad, err_in, beta1, len, bits_out, scale_out, err_out, part, st); break;
    case ONEBIT_F16: e = launch_vec<__half>(m, grad, err_in, beta1, len, bits_out, scale_out, err_out, part, st); break;
    default: e = launch_vec<__nv_bfloat16>(m, grad, err_in, beta1, len, bits_out, scale_out, err_out, part, st); break;
  }
  return e == cudaSuccess ? ONEBIT_OK : ONEBIT_ERR_CUDA;
}
