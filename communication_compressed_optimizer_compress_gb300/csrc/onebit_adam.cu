// onebit_adam.cu -- host side of the C ABI declared in include/onebit_adam.h.
//
// The handle owns: the chunk plan (the multi-tensor launcher's work tables: server-side chunks that
// never cross a server shard, and the worker kernel's chunks, which may hold several short shards),
// the workspace layout,
// the phase machine (warm-up -> freeze -> compression), the representation flags of the lazily
// materialised state (see onebit_kernels.cuh), a small ring of device-side gradient pointer tables,
// and optional per-kernel CUDA-event timing.  Every hot-path operation runs in the kernels.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/onebit_adam.h"
#include "onebit_kernels.cuh"

using namespace onebit;

namespace {

constexpr size_t kAlign = 256;
constexpr int kPtrRing = 4;
constexpr int kCopyStreams = 4;               // host-gradient copies run on this many internal streams
constexpr size_t kCopyPiece = size_t(64) << 20;  // and are cut into pieces of at most this size

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t round32(int64_t v) { return (v + 31) / 32 * 32; }
constexpr int64_t kMaxElements = int64_t(1) << 40;  // a parameter list's largest element count

struct Plan {
  int n = 0, T = 0;               // T: compressed segments (the tensors, or their scale blocks)
  std::vector<int64_t> numel;     // [T]
  int Tu = 0;                     // the caller's tensors
  std::vector<int64_t> unumel;    // [Tu]
  std::vector<int32_t> ufirst;    // [Tu+1]: segments of caller tensor k are ufirst[k] .. ufirst[k+1]-1
  std::vector<int64_t> voff;      // [T]: a segment's first element within its caller tensor
  bool split = false;             // scale_block > 0
  std::vector<int64_t> seg_off;   // padded offsets
  std::vector<int64_t> seg_uoff;  // unpadded offsets
  int64_t Dp = 0, D = 0, Wp = 0, Wr = 0;  // Wr: worker sign-row stride in words (multiple of 4)
  std::vector<Chunk> chunks;
  std::vector<Range> seg_ranges;    // [T]
  std::vector<Range> shard_ranges;  // [T*n]
  std::vector<Chunk> wchunks;       // worker-side chunks (never cross a tensor; may span shards)
  std::vector<Range> wseg_ranges;   // [T]
  int32_t max_wseg_count = 0, max_shard_count = 0;
  int32_t max_wchunk_len = 0;  // the longest worker-side chunk
  bool worker_spans = false;  // some worker chunk holds several shards
  bool contig = false;        // server kernels walk contiguous runs (see make_plan)
  // Multi-GPU form (make_rank_plan): rank `rank` of `world` holds the nl = n/world workers
  // w0 .. w0+nl-1 (w0 = rank*nl) and serves shards w0 .. w0+nl-1 of every segment.  One GPU
  // simulating all n workers is rank 0 of 1.
  int rank = 0, world = 1, nl = 0, w0 = 0;
  bool ranked = false;              // created by onebit_adam_init_rank: the exchange calls are legal
  std::vector<Chunk> schunks;       // this rank's server-side chunks (its shards), in plan order
  std::vector<Range> sshard_ranges; // [T*n] their ranges within schunks (count 0 for other ranks' shards)
  int64_t xsend = 0, xbcast = 0;    // words per exchange block: all-to-all, all-gather
  std::vector<XRange> xr[4];        // exchange copies of the four stages (see make_rank_plan)
  std::vector<int64_t> xrows[4];    // the same copies as host rows (onebit_adam_plan_exchange)
};

// Server shard j of a tensor of L elements: [j*S, min((j+1)*S, L)), S = 32*ceil(L/(32n)).
void shard_bounds(int64_t L, int n, int j, int64_t* lo, int64_t* hi) {
  const int64_t per = 32 * ((L + 32 * (int64_t)n - 1) / (32 * (int64_t)n));
  *lo = std::min<int64_t>((int64_t)j * per, L);
  *hi = std::min<int64_t>((int64_t)(j + 1) * per, L);
}

onebit_status_t check_config(const onebit_adam_config_t* cfg) {
  if (!cfg || !cfg->numel) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->n_workers < 1 || cfg->n_workers > kMaxWorkers) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->n_tensors < 1) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->grad_dtype < ONEBIT_F32 || cfg->grad_dtype > ONEBIT_BF16) return ONEBIT_ERR_INVALID_ARG;
  if (!(cfg->beta1 >= 0.0f && cfg->beta1 < 1.0f) || !(cfg->beta2 >= 0.0f && cfg->beta2 < 1.0f))
    return ONEBIT_ERR_INVALID_ARG;
  if (!(cfg->eps >= 0.0f) || !std::isfinite(cfg->eps) || !std::isfinite(cfg->lr)) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->warmup_steps < 1) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->bias_correction != 0 && cfg->bias_correction != 1) return ONEBIT_ERR_INVALID_ARG;
  if (cfg->scale_block < 0 || cfg->scale_block % 32 != 0) return ONEBIT_ERR_INVALID_ARG;
  int64_t total = 0;
  for (int k = 0; k < cfg->n_tensors; ++k) {
    if (cfg->numel[k] < 0) return ONEBIT_ERR_INVALID_ARG;
    total += cfg->numel[k];
  }
  if (total < 1) return ONEBIT_ERR_INVALID_ARG;
  if (total > kMaxElements) return ONEBIT_ERR_UNSUPPORTED;  // far beyond any device's memory
  return ONEBIT_OK;
}

// The multi-tensor launcher's table: chunks of at most chunk_length() elements that never cross a tensor
// or a server-shard boundary.  Shard boundaries are multiples of 32 inside a tensor, so every chunk
// starts on a sign-word boundary and only a tensor's last chunk can have a ragged end.
// Chunk length: kChunk for large lists; shorter (a multiple of 4096) for small ones, so that even a
// small list yields about kChunkTarget work units.  It depends on the element count only, never on
// the device, so results do not depend on the GPU they run on.
constexpr int64_t kChunkTarget = 1216;
int64_t chunk_length(int64_t total) {
  const int64_t want = (total + kChunkTarget - 1) / kChunkTarget;
  return std::min<int64_t>(kChunk, std::max<int64_t>(4096, (want + 4095) / 4096 * 4096));
}

onebit_status_t make_plan(const onebit_adam_config_t* cfg, Plan* P) {
  P->n = cfg->n_workers;
  P->Tu = cfg->n_tensors;
  P->unumel.assign(cfg->numel, cfg->numel + cfg->n_tensors);
  P->split = cfg->scale_block > 0;
  // Segments: with a scale block B, tensor k is cut into ceil(L_k/B) blocks (an empty tensor keeps
  // one empty block) and every block is compressed as a tensor of its own.
  int64_t total = 0;
  P->ufirst.assign(1, 0);
  for (int k = 0; k < P->Tu; ++k) {
    const int64_t L = P->unumel[k];
    total += L;
    const int64_t B = P->split ? cfg->scale_block : std::max<int64_t>(L, 1);
    const int64_t blocks = L > 0 ? (L + B - 1) / B : 1;
    // checked before anything is built: a tiny block on a huge tensor must not exhaust host memory
    if (((int64_t)P->numel.size() + blocks) * P->n > (int64_t)INT32_MAX) return ONEBIT_ERR_UNSUPPORTED;
    int64_t s = 0;
    do {
      P->numel.push_back(std::min<int64_t>(B, L - s));
      P->voff.push_back(s);
      s += B;
    } while (s < L);
    P->ufirst.push_back((int32_t)P->numel.size());
  }
  P->T = (int)P->numel.size();
  const int64_t clen = chunk_length(total);
  P->seg_off.resize(P->T);
  P->seg_uoff.resize(P->T);
  P->seg_ranges.resize(P->T);
  P->wseg_ranges.resize(P->T);
  P->shard_ranges.resize((size_t)P->T * P->n);
  int64_t off = 0, uoff = 0;
  for (int k = 0; k < P->T; ++k) {
    const int64_t L = P->numel[k];
    P->seg_off[k] = off;
    P->seg_uoff[k] = uoff;
    Range sr{(int32_t)P->chunks.size(), 0, L};
    for (int j = 0; j < P->n; ++j) {
      int64_t lo, hi;
      shard_bounds(L, P->n, j, &lo, &hi);
      Range hr{(int32_t)P->chunks.size(), 0, hi - lo};
      for (int64_t s = lo; s < hi; s += clen) {
        Chunk c{};
        c.off = off + s;
        c.uoff = uoff + s;
        c.start = s;
        c.seg = k;
        c.shard = j;
        c.len = (int32_t)std::min<int64_t>(clen, hi - s);
        P->chunks.push_back(c);
        if (P->chunks.size() > (size_t)INT32_MAX) return ONEBIT_ERR_UNSUPPORTED;
      }
      hr.count = (int32_t)P->chunks.size() - hr.first;
      P->shard_ranges[(size_t)k * P->n + j] = hr;
    }
    sr.count = (int32_t)P->chunks.size() - sr.first;
    P->seg_ranges[k] = sr;
    // Worker-side chunks.  With shards at least a chunk long they are the server-side chunks.  With
    // shorter shards a worker chunk holds as many whole shards as fit in chunk_length() elements, so
    // that the worker kernel's units stay long; such a chunk records the shard length, and each of
    // its groups finds its own shard from its offset inside the chunk.
    const int64_t per = 32 * ((L + 32 * (int64_t)P->n - 1) / (32 * (int64_t)P->n));
    Range wr{(int32_t)P->wchunks.size(), 0, L};
    if (per >= clen) {
      P->wchunks.insert(P->wchunks.end(), P->chunks.begin() + sr.first, P->chunks.begin() + sr.first + sr.count);
    } else if (L > 0) {
      const int64_t step = clen / per * per;
      for (int64_t s = 0; s < L; s += step) {
        Chunk c{};
        c.off = off + s;
        c.uoff = uoff + s;
        c.start = s;
        c.seg = k;
        c.len = (int32_t)std::min<int64_t>(step, L - s);
        c.shard = (int32_t)(s / per);
        c.per = c.len > per ? (int32_t)per : 0;
        P->wchunks.push_back(c);
      }
    }
    if (P->wchunks.size() > (size_t)INT32_MAX) return ONEBIT_ERR_UNSUPPORTED;
    wr.count = (int32_t)P->wchunks.size() - wr.first;
    P->wseg_ranges[k] = wr;
    P->max_wseg_count = std::max(P->max_wseg_count, wr.count);
    for (int j = 0; j < P->n; ++j)
      P->max_shard_count = std::max(P->max_shard_count, P->shard_ranges[(size_t)k * P->n + j].count);
    off += round32(L);
    uoff += L;
  }
  P->Dp = off;
  P->D = uoff;
  for (const Chunk& c : P->wchunks) {
    P->worker_spans |= c.per != 0;
    P->max_wchunk_len = std::max(P->max_wchunk_len, c.len);
  }
  // The server rebuilds its sum tables (about 2^min(n,12) entries) whenever a CTA moves to another
  // tensor.  Striding over the chunks, that happens at nearly every chunk once tensors are shorter
  // than a grid's worth of chunks.  When those rebuilds would cost more than about 5% of the
  // elements, the server kernel walks contiguous runs of chunks instead (both of its variants).
  const int64_t table = (int64_t(1) << std::min(P->n, 12)) + (P->n > 12 ? 512 : 0);
  P->contig = P->T > 1 && table * (int64_t)P->chunks.size() * 20 > P->D;
  P->Wp = off / 32;
  P->Wr = (P->Wp + 3) / 4 * 4;
  P->nl = P->n;  // one GPU simulating every worker; make_rank_plan() narrows it
  return ONEBIT_OK;
}

// Words of segment k's sign words that hold the shards of rank q: [lo, hi) in the segment's word
// space (shard boundaries are multiples of 32 inside a segment; the last word may hold padding bits).
void rank_words(const Plan& P, int k, int q, int64_t* lo, int64_t* hi) {
  int64_t a, b, c, d;
  shard_bounds(P.numel[k], P.n, q * P.nl, &a, &b);
  shard_bounds(P.numel[k], P.n, (q + 1) * P.nl - 1, &c, &d);
  *lo = a / 32;
  *hi = d > a ? (d + 31) / 32 : a / 32;
}

// The multi-GPU form's partition and exchange copies.  Regions: 0 worker sign rows (row = worker,
// word in the padded word layout), 1 worker scales (row = worker, column = segment), 2 server sign
// words (row 0), 3 server scales (row = segment, column = shard), 4 the caller's exchange buffer
// (row = block, i.e. rank).  Stages:
//   0 (begin)  pack, into block q of the all-to-all send buffer, every local worker's scales and the
//              sign words of rank q's shards: per local worker il, T scales then the words, segment
//              by segment (worker il's part of block q starts at il*(T + Wq), Wq = words of q's shards);
//   1 (serve)  unpack block p of the received buffer into the rows of rank p's workers;
//   2 (serve)  pack this rank's server scales (segment-major, nl per segment) and the server sign
//              words of its shards into its all-gather block;
//   3 (end)    unpack every other rank's all-gather block into the server scales and sign words.
// A rank's own block is never copied: its data is already in place.
onebit_status_t make_rank_plan(Plan* P, int rank, int world) {
  P->rank = rank;
  P->world = world;
  P->nl = P->n / world;
  P->w0 = rank * P->nl;
  const int T = P->T, n = P->n, nl = P->nl;
  // this rank's server-side chunks, with shard ranges relative to them
  P->schunks.clear();
  P->sshard_ranges.assign((size_t)T * n, Range{0, 0, 0});
  for (int k = 0; k < T; ++k)
    for (int j = 0; j < n; ++j) {
      const Range g = P->shard_ranges[(size_t)k * n + j];
      Range r{(int32_t)P->schunks.size(), 0, g.len};
      if (j >= P->w0 && j < P->w0 + nl) {
        P->schunks.insert(P->schunks.end(), P->chunks.begin() + g.first, P->chunks.begin() + g.first + g.count);
        r.count = g.count;
      }
      P->sshard_ranges[(size_t)k * n + j] = r;
    }
  // words of each rank's shards, per segment, and their prefix sums
  std::vector<int64_t> wlo((size_t)world * T), whi((size_t)world * T), cum((size_t)world * (T + 1), 0);
  int64_t wmax = 0;
  for (int q = 0; q < world; ++q) {
    for (int k = 0; k < T; ++k) {
      rank_words(*P, k, q, &wlo[(size_t)q * T + k], &whi[(size_t)q * T + k]);
      cum[(size_t)q * (T + 1) + k + 1] = cum[(size_t)q * (T + 1) + k] + whi[(size_t)q * T + k] - wlo[(size_t)q * T + k];
    }
    wmax = std::max(wmax, cum[(size_t)q * (T + 1) + T]);
  }
  P->xsend = (int64_t)nl * (T + wmax);
  P->xbcast = (int64_t)T * nl + wmax;
  for (int st = 0; st < 4; ++st) {
    P->xr[st].clear();
    P->xrows[st].clear();
  }
  const int64_t row_stride[5] = {P->Wr, T, 0, n, 0};
  auto add = [&](int st, int sreg, int64_t srow, int64_t soff, int dreg, int64_t drow, int64_t doff, int64_t len) {
    if (len <= 0) return;
    const int64_t block = st < 2 ? P->xsend : P->xbcast;
    const int64_t s0 = (sreg == 4 ? srow * block : srow * row_stride[sreg]) + soff;
    const int64_t d0 = (dreg == 4 ? drow * block : drow * row_stride[dreg]) + doff;
    const int64_t r[8] = {st, sreg, srow, soff, dreg, drow, doff, len};
    P->xrows[st].insert(P->xrows[st].end(), r, r + 8);
    for (int64_t o = 0; o < len; o += kXPiece)
      P->xr[st].push_back(XRange{s0 + o, d0 + o, (int32_t)std::min<int64_t>(kXPiece, len - o), (int16_t)sreg,
                                 (int16_t)dreg});
  };
  auto seg_word = [&](int k) { return P->seg_off[k] / 32; };
  const int64_t Wme = cum[(size_t)rank * (T + 1) + T];
  for (int q = 0; q < world; ++q) {
    if (q == rank) continue;
    const int64_t Wq = cum[(size_t)q * (T + 1) + T];
    for (int il = 0; il < nl; ++il) {
      const int w = P->w0 + il;  // stage 0: this rank's worker w, for rank q's shards
      add(0, 1, w, 0, 4, q, (int64_t)il * (T + Wq), T);
      for (int k = 0; k < T; ++k)
        add(0, 0, w, seg_word(k) + wlo[(size_t)q * T + k], 4, q, (int64_t)il * (T + Wq) + T + cum[(size_t)q * (T + 1) + k],
            whi[(size_t)q * T + k] - wlo[(size_t)q * T + k]);
      const int wp = q * nl + il;  // stage 1: rank q's worker wp, for this rank's shards
      add(1, 4, q, (int64_t)il * (T + Wme), 1, wp, 0, T);
      for (int k = 0; k < T; ++k)
        add(1, 4, q, (int64_t)il * (T + Wme) + T + cum[(size_t)rank * (T + 1) + k], 0, wp,
            seg_word(k) + wlo[(size_t)rank * T + k], whi[(size_t)rank * T + k] - wlo[(size_t)rank * T + k]);
    }
    // stage 3: rank q's server scales and sign words
    for (int k = 0; k < T; ++k) add(3, 4, q, (int64_t)k * nl, 3, k, (int64_t)q * nl, nl);
    for (int k = 0; k < T; ++k)
      add(3, 4, q, (int64_t)T * nl + cum[(size_t)q * (T + 1) + k], 2, 0, seg_word(k) + wlo[(size_t)q * T + k],
          whi[(size_t)q * T + k] - wlo[(size_t)q * T + k]);
  }
  if (world > 1) {  // stage 2: this rank's block of the all-gather
    for (int k = 0; k < T; ++k) add(2, 3, k, P->w0, 4, 0, (int64_t)k * nl, nl);
    for (int k = 0; k < T; ++k)
      add(2, 2, 0, seg_word(k) + wlo[(size_t)rank * T + k], 4, 0, (int64_t)T * nl + cum[(size_t)rank * (T + 1) + k],
          whi[(size_t)rank * T + k] - wlo[(size_t)rank * T + k]);
  }
  for (int st = 0; st < 4; ++st)
    if (P->xr[st].size() > (size_t)INT32_MAX) return ONEBIT_ERR_UNSUPPORTED;
  return ONEBIT_OK;
}

struct Layout {
  size_t m, v, a, c, wbits, sbits, wscale, sscale, wpart, spart, chunks, seg_ranges, shard_ranges, wchunks,
      wseg_ranges, schunks, sshard_ranges, xr[4], gptr, pptr, status, total;
};

Layout make_layout(const Plan& P) {
  Layout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1), kAlign);
    return at;
  };
  const size_t n = P.n, nl = P.nl, T = P.T, C = P.chunks.size();
  L.m = take(P.Dp * 4);
  L.v = take(P.Dp * 4);
  L.a = take(P.Dp * 4);
  L.c = take(nl * P.Dp * 4);  // only this rank's workers keep c
  L.wbits = take(n * P.Wr * 4);
  L.sbits = take(P.Wp * 4);
  L.wscale = take(2 * n * T * 4);
  L.sscale = take(2 * n * T * 4);
  L.wpart = take(nl * P.wchunks.size() * 8);
  L.spart = take(C * 8);
  // host-built tables, uploaded together (chunks .. xr[3])
  L.chunks = take(C * sizeof(Chunk));
  L.seg_ranges = take(T * sizeof(Range));
  L.shard_ranges = take(T * n * sizeof(Range));
  L.wchunks = take(P.wchunks.size() * sizeof(Chunk));
  L.wseg_ranges = take(T * sizeof(Range));
  L.schunks = take(P.schunks.size() * sizeof(Chunk));
  L.sshard_ranges = take(P.sshard_ranges.size() * sizeof(Range));
  for (int st = 0; st < 4; ++st) L.xr[st] = take(P.xr[st].size() * sizeof(XRange));
  L.gptr = take(kPtrRing * n * T * sizeof(void*));
  L.pptr = take(T * sizeof(void*));
  L.status = take(256);
  L.total = o;
  return L;
}

struct TimedLaunch {
  int kernel;
  cudaEvent_t start, stop;
};

}  // namespace

struct onebit_adam {
  onebit_adam_config_t cfg{};
  Plan plan;
  Layout lay{};
  int device = 0;
  int num_sms = 0;
  uint8_t* ws = nullptr;
  bool ws_owned = false;
  std::vector<float*> params;
  bool params_aligned = true;
  // phase machine
  int64_t t = 0;
  int32_t phase = ONEBIT_PHASE_WARMUP;
  int64_t compress_steps = 0;  // parity of the scale buffers
  bool m_dense = true;
  bool werr_zero = true;
  bool serr_zero = true;
  // gradient pointer table ring
  std::vector<std::vector<const void*>> ring;
  std::vector<const void*> gexp;  // per-segment gradient pointers of the current step (scale blocks)
  int ring_next = 0;
  // host-gradient staging: two device buffers used alternately, so that one step's copies can run
  // while the previous step's kernels still read the other buffer
  uint8_t* staging[2] = {nullptr, nullptr};
  int stage_next = 0;
  cudaStream_t copy_st[kCopyStreams] = {};
  cudaEvent_t ev_copied[kCopyStreams] = {};
  cudaEvent_t ev_free[2] = {};  // recorded after the last step that read staging[i]
  bool ev_free_recorded[2] = {false, false};
  // timing
  bool timing = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> event_pool;
  int64_t launches = 0;
  std::unordered_map<const void*, int> occupancy;
  std::unordered_set<const void*> dyn_smem_set;  // kernels whose dynamic shared-memory limit is raised
  uint32_t stall_tx = 0;  // fault injection (see onebit_adam_set_fault_injection)
  int64_t check_margin = 0;  // checked builds: padded elements the bounds checks withhold (test hook)
  int fail_allocs = 0;    // allocations still to refuse (fault injection)
  int max_ctas = 0;       // cap on the CTAs of a streaming launch (0: fill the GPU)
  // variance-norm monitor (warm-up)
  bool vmon = false;
  double* vnorm_host = nullptr;  // pinned
  cudaEvent_t ev_vnorm = nullptr;
  int64_t vnorm_step = 0;
  // automatic freeze: tolerance on the norm's relative change per step (0: off), last norm seen
  double auto_tol = 0.0;
  bool auto_have_prev = false;
  double auto_prev = 0.0;
  std::string last_error;
  int xstage = 0;  // multi-GPU form: 0 idle, 1 after compress_begin, 2 after compress_serve

  template <typename T> T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
};

namespace {

// Tracing: every public step and state call is one named NVTX range (visible in Nsight tools;
// a no-op when no tool is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Fault injection: true when this allocation is to be refused (ONEBIT_FAULT_FAIL_ALLOC).
bool refuse_alloc(onebit_adam* h) {
  if (h->fail_allocs <= 0) return false;
  --h->fail_allocs;
  return true;
}

onebit_status_t cuda_fail(onebit_adam* h, cudaError_t e, const char* where) {
  if (h) h->last_error = std::string(where) + ": " + cudaGetErrorString(e);
  return ONEBIT_ERR_CUDA;
}

// The pinned host slot (and its event) that receives the variance norm of monitored warm-up steps.
onebit_status_t ensure_vnorm_slot(onebit_adam* h) {
  if (h->vnorm_host) return ONEBIT_OK;
  if (refuse_alloc(h) ||
      cudaHostAlloc(reinterpret_cast<void**>(&h->vnorm_host), sizeof(double), cudaHostAllocDefault) != cudaSuccess) {
    cudaGetLastError();
    h->vnorm_host = nullptr;
    return ONEBIT_ERR_NOMEM;
  }
  *h->vnorm_host = 0.0;
  if (cudaEventCreateWithFlags(&h->ev_vnorm, cudaEventDisableTiming) != cudaSuccess) {
    const cudaError_t e = cudaGetLastError();
    cudaFreeHost(h->vnorm_host);
    h->vnorm_host = nullptr;
    return cuda_fail(h, e, "cudaEventCreateWithFlags");
  }
  return ONEBIT_OK;
}

// The CUDA message of the last onebit_adam_init that failed on this thread: its handle is gone, so
// onebit_adam_last_error(NULL) returns this.
thread_local std::string t_init_error;

#define ONEBIT_CUDA(h, call)                                  \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return cuda_fail((h), e_, #call);  \
  } while (0)

cudaStream_t as_stream(onebit_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

int grid_for(onebit_adam* h, const void* fn, int threads, int64_t units, size_t dyn_smem = 0) {
  auto it = h->occupancy.find(fn);
  int per_sm;
  if (it == h->occupancy.end()) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, dyn_smem) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    h->occupancy[fn] = per_sm;
  } else {
    per_sm = it->second;
  }
  int64_t g = std::min<int64_t>(units, (int64_t)h->num_sms * per_sm);
  if (h->max_ctas > 0) g = std::min<int64_t>(g, h->max_ctas);
  return (int)std::max<int64_t>(1, g);
}

cudaEvent_t take_event(onebit_adam* h) {
  if (!h->event_pool.empty()) {
    cudaEvent_t e = h->event_pool.back();
    h->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Launch one kernel on `stream`, bracketed by timing events when timing is on.
template <typename Kern, typename Arg>
onebit_status_t launch(onebit_adam* h, int kid, Kern kern, int grid, int threads, cudaStream_t stream,
                       const Arg& arg, size_t dyn_smem = 0) {
  TimedLaunch tl{kid, nullptr, nullptr};
  if (h->timing) {
    tl.start = take_event(h);
    tl.stop = take_event(h);
    if (tl.start) cudaEventRecord(tl.start, stream);
  }
  kern<<<grid, threads, dyn_smem, stream>>>(arg);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(h, e, "kernel launch");
  ++h->launches;
  if (h->timing && tl.start && tl.stop) {
    cudaEventRecord(tl.stop, stream);
    h->timed.push_back(tl);
  }
  return ONEBIT_OK;
}

StepArgs base_args(onebit_adam* h) {
  const Plan& P = h->plan;
  const Layout& L = h->lay;
  StepArgs A{};
  A.chunks = h->at<Chunk>(L.chunks);
  A.n_chunks = (int32_t)P.chunks.size();
  A.wchunks = h->at<Chunk>(L.wchunks);
  A.n_wchunks = (int32_t)P.wchunks.size();
  A.wseg_ranges = h->at<Range>(L.wseg_ranges);
  A.n = P.n;
  A.T = P.T;
  A.pow2 = (P.n & (P.n - 1)) == 0;
  A.Dp = P.Dp;
  A.D = P.D;
  A.contig = P.contig ? 1 : 0;
  A.Wp = P.Wp;
  A.Wr = P.Wr;
  A.pptr = h->at<float*>(L.pptr);
  A.m = h->at<float>(L.m);
  A.v = h->at<float>(L.v);
  A.c = h->at<float>(L.c);
  A.a = h->at<float>(L.a);
  A.wbits = h->at<uint32_t>(L.wbits);
  A.sbits = h->at<uint32_t>(L.sbits);
  const int cur = (int)(h->compress_steps & 1), prev = cur ^ 1;
  const size_t nt = (size_t)P.n * P.T;
  A.wscale_prev = h->at<float>(L.wscale) + prev * nt;
  A.wscale_cur = h->at<float>(L.wscale) + cur * nt;
  A.sscale_prev = h->at<float>(L.sscale) + prev * nt;
  A.sscale_cur = h->at<float>(L.sscale) + cur * nt;
  A.wpart = h->at<double>(L.wpart);
  A.spart = h->at<double>(L.spart);
  A.seg_ranges = h->at<Range>(L.seg_ranges);
  A.shard_ranges = h->at<Range>(L.shard_ranges);
  A.status = h->at<unsigned int>(L.status);
  const onebit_adam_config_t& c = h->cfg;
  A.b1 = c.beta1;
  A.omb1 = 1.0f - c.beta1;  // fp32 arithmetic, as the method's constants are fp32
  A.b2 = c.beta2;
  A.omb2 = 1.0f - c.beta2;
  A.lr = c.lr;
  A.eps = c.eps;
  A.nf = (float)P.n;
  A.inv_n = 1.0f / (float)P.n;
  A.bc1 = 1.0f;
  A.bc2 = 1.0f;
  A.stall_tx = h->stall_tx;
  A.nl = P.nl;
  A.w0 = P.w0;
#ifdef ONEBIT_CHECKS
  A.check_margin = h->check_margin;
#endif
  return A;
}

// The server kernels of the multi-GPU form run over this rank's shards only.
void narrow_to_own_shards(const onebit_adam* h, StepArgs* A) {
  if (!h->plan.ranked) return;
  A->chunks = h->at<Chunk>(h->lay.schunks);
  A->n_chunks = (int32_t)h->plan.schunks.size();
  A->shard_ranges = h->at<Range>(h->lay.sshard_ranges);
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Upload (or reuse) the [n*T] gradient pointer table; reports whether every gradient pointer allows
// the vector loads of the kernels.
onebit_status_t bind_grads(onebit_adam* h, const void* const* grads, int nw, cudaStream_t stream,
                           const void* const** dev, bool* vec) {
  const Plan& P = h->plan;
  const size_t cnt = (size_t)nw * P.T;  // nw: the workers whose gradients are passed (n, or a rank's nl)
  const size_t gb = h->cfg.grad_dtype == ONEBIT_F32 ? 4 : 2;
  for (size_t q = 0; q < (size_t)nw * P.Tu; ++q)
    if (!grads[q] && P.unumel[q % P.Tu] > 0) return ONEBIT_ERR_INVALID_ARG;
  if (P.split) {  // one pointer per segment: its caller tensor's pointer advanced to the block
    h->gexp.resize(cnt);
    for (int i = 0; i < nw; ++i)
      for (int k = 0; k < P.Tu; ++k) {
        const uint8_t* g = static_cast<const uint8_t*>(grads[(size_t)i * P.Tu + k]);
        for (int v = P.ufirst[k]; v < P.ufirst[k + 1]; ++v)
          h->gexp[(size_t)i * P.T + v] = g ? g + P.voff[v] * gb : nullptr;
      }
    grads = h->gexp.data();
  }
  const size_t galign = gb == 4 ? 32 : 16;
  bool ok = true;
  for (size_t q = 0; q < cnt; ++q)
    if (!aligned(grads[q], galign)) ok = false;
  *vec = ok;
  const void** base = h->at<const void*>(h->lay.gptr);
  for (int r = 0; r < kPtrRing; ++r) {
    if (h->ring[r].size() == cnt && std::equal(h->ring[r].begin(), h->ring[r].end(), grads)) {
      *dev = base + (size_t)r * cnt;
      return ONEBIT_OK;
    }
  }
  const int r = h->ring_next;
  h->ring_next = (h->ring_next + 1) % kPtrRing;
  h->ring[r].assign(grads, grads + cnt);
  ONEBIT_CUDA(h, cudaMemcpyAsync(base + (size_t)r * cnt, h->ring[r].data(), cnt * sizeof(void*),
                                 cudaMemcpyHostToDevice, stream));
  *dev = base + (size_t)r * cnt;
  return ONEBIT_OK;
}

template <typename GT, bool MON>
onebit_status_t run_warmup_m(onebit_adam* h, const StepArgs& A, bool vec, cudaStream_t st) {
  const int C = A.n_chunks;
  const bool bc = h->cfg.bias_correction != 0;
  if constexpr (sizeof(GT) == 2) {
    if (vec && A.n >= kWarmStagedMin && A.n <= kWarmStagedMax) {
      // many 16-bit gradient streams: the shared-memory staged variant keeps enough bytes in flight
      const size_t dyn = warmup_dyn_smem(A.n);
      auto go = [&](auto kern) -> onebit_status_t {
        if (!h->dyn_smem_set.count((const void*)kern)) {
          cudaError_t e = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)warmup_dyn_smem(kWarmStagedMax));
          if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute");
          h->dyn_smem_set.insert((const void*)kern);
        }
        return launch(h, ONEBIT_K_WARMUP, kern, grid_for(h, (const void*)kern, kStagedThreads, C, dyn), kStagedThreads,
                      st, A, dyn);
      };
      return bc ? go(k_warmup_staged<GT, true, MON>) : go(k_warmup_staged<GT, false, MON>);
    }
  }
  auto pick = [&](auto kern) { return launch(h, ONEBIT_K_WARMUP, kern, grid_for(h, (const void*)kern, kThreads, C), kThreads, st, A); };
  if constexpr (sizeof(GT) == 2) {  // 16-bit gradients, all in one small batch (measured slower for fp32)
    if (A.n <= 4) {
      if (bc) return vec ? pick(k_warmup<GT, true, true, MON, true>) : pick(k_warmup<GT, true, false, MON, true>);
      return vec ? pick(k_warmup<GT, false, true, MON, true>) : pick(k_warmup<GT, false, false, MON, true>);
    }
  }
  if (bc) return vec ? pick(k_warmup<GT, true, true, MON, false>) : pick(k_warmup<GT, true, false, MON, false>);
  return vec ? pick(k_warmup<GT, false, true, MON, false>) : pick(k_warmup<GT, false, false, MON, false>);
}

// warm-up steps compute the variance norm for the monitor and for the automatic freeze
bool monitored(const onebit_adam* h) { return h->vmon || h->auto_tol > 0.0; }

template <typename GT>
onebit_status_t run_warmup(onebit_adam* h, StepArgs A, bool vec, cudaStream_t st) {
  return monitored(h) ? run_warmup_m<GT, true>(h, A, vec, st) : run_warmup_m<GT, false>(h, A, vec, st);
}

template <typename GT, int DM, bool HE>
onebit_status_t run_worker_v(onebit_adam* h, const StepArgs& A, bool vec, cudaStream_t st) {
  const int64_t units = (int64_t)A.n_wchunks * A.nl;
  if constexpr (DM == kMomBits || DM == kMomBitsShards) {
    // short units, and enough of them to give every SM 32 warps: one warp each
    if (h->plan.max_wchunk_len <= kWarpUnitMax && units >= (int64_t)32 * h->num_sms) {
      const int64_t blocks = (units + kThreads / 32 - 1) / (kThreads / 32);
      auto k = vec ? k_worker<GT, DM, HE, true, true> : k_worker<GT, DM, HE, false, true>;
      return launch(h, ONEBIT_K_WORKER, k, grid_for(h, (const void*)k, kThreads, blocks), kThreads, st, A);
    }
  }
  if (vec) {
    auto k = k_worker<GT, DM, HE, true>;
    return launch(h, ONEBIT_K_WORKER, k, grid_for(h, (const void*)k, kThreads, units), kThreads, st, A);
  }
  auto k = k_worker<GT, DM, HE, false>;
  return launch(h, ONEBIT_K_WORKER, k, grid_for(h, (const void*)k, kThreads, units), kThreads, st, A);
}

template <typename GT>
onebit_status_t run_worker(onebit_adam* h, const StepArgs& A, bool vec, cudaStream_t st, bool grad_only) {
  const bool he = !h->werr_zero;
  if (grad_only) return he ? run_worker_v<GT, kMomNone, true>(h, A, vec, st) : run_worker_v<GT, kMomNone, false>(h, A, vec, st);
  if (h->m_dense) return he ? run_worker_v<GT, kMomDense, true>(h, A, vec, st) : run_worker_v<GT, kMomDense, false>(h, A, vec, st);
  if (h->plan.worker_spans)
    return he ? run_worker_v<GT, kMomBitsShards, true>(h, A, vec, st) : run_worker_v<GT, kMomBitsShards, false>(h, A, vec, st);
  return he ? run_worker_v<GT, kMomBits, true>(h, A, vec, st) : run_worker_v<GT, kMomBits, false>(h, A, vec, st);
}

template <bool HE, bool CONTIG>
onebit_status_t run_server_staged(onebit_adam* h, const StepArgs& A, cudaStream_t st) {
  // shared-memory staged variant: the tiles of a and the n sign rows arrive by bulk copies; the
  // common worker counts have their own compile-time instances
  auto go = [&](auto k) -> onebit_status_t {
    const size_t dyn = server_dyn_smem(A.n);
    if (!h->dyn_smem_set.count((const void*)k)) {
      cudaError_t e = cudaFuncSetAttribute((const void*)k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)server_dyn_smem(kStageMaxWorkers));
      if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute");
      h->dyn_smem_set.insert((const void*)k);
    }
    return launch(h, ONEBIT_K_SERVER, k, grid_for(h, (const void*)k, kStagedThreads, A.n_chunks, dyn),
                  kStagedThreads, st, A, dyn);
  };
  switch (A.n) {
    case 4: return go(k_server_staged<HE, 4, CONTIG>);
    case 8: return go(k_server_staged<HE, 8, CONTIG>);
    case 16: return go(k_server_staged<HE, 16, CONTIG>);
    default: return go(k_server_staged<HE, 0, CONTIG>);
  }
}

template <bool HE>
onebit_status_t run_server_v(onebit_adam* h, const StepArgs& A, cudaStream_t st) {
  // CONTIG (many short tensors or scale blocks): contiguous runs of chunks, so that the sum tables
  // are rebuilt once per segment and CTA
  if (A.n <= kStageMaxWorkers)
    return A.contig ? run_server_staged<HE, true>(h, A, st) : run_server_staged<HE, false>(h, A, st);
  // register variant for larger n
  if (A.contig) {
    auto k = k_server<HE, true>;
    return launch(h, ONEBIT_K_SERVER, k, grid_for(h, (const void*)k, kThreads, A.n_chunks), kThreads, st, A);
  }
  auto k = k_server<HE, false>;
  return launch(h, ONEBIT_K_SERVER, k, grid_for(h, (const void*)k, kThreads, A.n_chunks), kThreads, st, A);
}

onebit_status_t run_server(onebit_adam* h, const StepArgs& A, cudaStream_t st) {
  return h->serr_zero ? run_server_v<false>(h, A, st) : run_server_v<true>(h, A, st);
}

// The broadcast and update over the whole replica.  Plans whose worker chunks hold several whole
// shards (short scale blocks) walk those: the units stay long, and each group finds its own shard.
onebit_status_t run_update(onebit_adam* h, const StepArgs& A, cudaStream_t st) {
  auto go = [&](auto k, int units) {
    return launch(h, ONEBIT_K_UPDATE, k, grid_for(h, (const void*)k, kThreads, units), kThreads, st, A);
  };
  if (h->plan.worker_spans)
    return h->params_aligned ? go(k_update<true, true>, A.n_wchunks) : go(k_update<false, true>, A.n_wchunks);
  return h->params_aligned ? go(k_update<true, false>, A.n_chunks) : go(k_update<false, false>, A.n_chunks);
}

// den = sqrt(v) + eps in place (v / (1 - b2^t) first with bias correction); the compression stage
// starts from zero errors and the dense warm-up momentum.
onebit_status_t do_freeze(onebit_adam* h, cudaStream_t st) {
  const int64_t groups = h->plan.Dp / 8;
  const float bc2 = (float)(1.0 - std::pow((double)h->cfg.beta2, (double)h->t));
  float* v = h->at<float>(h->lay.v);
  auto go = [&](auto kern) -> onebit_status_t {
    TimedLaunch tl{ONEBIT_K_FREEZE, nullptr, nullptr};
    if (h->timing) {
      tl.start = take_event(h);
      tl.stop = take_event(h);
      if (tl.start) cudaEventRecord(tl.start, st);
    }
    const int grid = grid_for(h, (const void*)kern, kThreads, (groups + kThreads - 1) / kThreads);
    kern<<<grid, kThreads, 0, st>>>(v, groups, bc2, h->cfg.eps);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "freeze launch");
    ++h->launches;
    if (h->timing && tl.start && tl.stop) {
      cudaEventRecord(tl.stop, st);
      h->timed.push_back(tl);
    }
    return ONEBIT_OK;
  };
  const onebit_status_t s = h->cfg.bias_correction ? go(k_freeze<true>) : go(k_freeze<false>);
  if (s) return s;
  h->phase = ONEBIT_PHASE_COMPRESS;
  h->m_dense = true;
  h->werr_zero = true;
  h->serr_zero = true;
  h->auto_have_prev = false;
  return ONEBIT_OK;
}

onebit_status_t do_warmup(onebit_adam* h, const void* const* grads, cudaStream_t st) {
  if (h->phase != ONEBIT_PHASE_WARMUP) return ONEBIT_ERR_PHASE;
  if (h->t >= h->cfg.warmup_steps) return ONEBIT_ERR_PHASE;
  StepArgs A = base_args(h);
  bool vec = false;
  onebit_status_t s = bind_grads(h, grads, h->plan.n, st, &A.gptr, &vec);  // every worker's gradient
  if (s) return s;
  const int64_t t = h->t + 1;
  A.bc1 = (float)(1.0 - std::pow((double)h->cfg.beta1, (double)t));
  A.bc2 = (float)(1.0 - std::pow((double)h->cfg.beta2, (double)t));
  vec = vec && h->params_aligned;
  switch (h->cfg.grad_dtype) {
    case ONEBIT_F32: s = run_warmup<float>(h, A, vec, st); break;
    case ONEBIT_F16: s = run_warmup<__half>(h, A, vec, st); break;
    default: s = run_warmup<__nv_bfloat16>(h, A, vec, st); break;
  }
  if (s) return s;
  h->t = t;
  if (monitored(h)) {  // ||v_t|| from the chunk partials, then to the pinned host slot
    double* slot = reinterpret_cast<double*>(h->ws + h->lay.status + 64);
    k_variance_norm<<<1, kScaleThreads, 0, st>>>(h->at<double>(h->lay.spart), A.n_chunks, slot);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(h, e, "variance norm launch");
    ++h->launches;
    ONEBIT_CUDA(h, cudaMemcpyAsync(h->vnorm_host, slot, sizeof(double), cudaMemcpyDeviceToHost, st));
    ONEBIT_CUDA(h, cudaEventRecord(h->ev_vnorm, st));
    h->vnorm_step = t;
  }
  if (h->auto_tol > 0.0) {
    // the automatic freeze: the variance norm's relative change per step against the tolerance
    ONEBIT_CUDA(h, cudaEventSynchronize(h->ev_vnorm));
    const double cur = *h->vnorm_host;
    const bool stable = h->auto_have_prev && std::fabs(cur - h->auto_prev) <= h->auto_tol * h->auto_prev;
    h->auto_prev = cur;
    h->auto_have_prev = true;
    if (stable || t >= h->cfg.warmup_steps) return do_freeze(h, st);
  }
  return ONEBIT_OK;
}

// One compression-stage step, or (ec_adam) one step of the gradient-compression baseline: the
// same worker/server compression of g_i + delta_i, then Adam on the broadcast.
// The worker half of a step: K1 for the handle's workers (all n, or a rank's nl) and their scales.
onebit_status_t run_worker_half(onebit_adam* h, const void* const* grads, cudaStream_t st, bool ec_adam) {
  StepArgs A = base_args(h);
  bool vec = false;
  onebit_status_t s = bind_grads(h, grads, h->plan.nl, st, &A.gptr, &vec);
  if (s) return s;
  switch (h->cfg.grad_dtype) {
    case ONEBIT_F32: s = run_worker<float>(h, A, vec, st, ec_adam); break;
    case ONEBIT_F16: s = run_worker<__half>(h, A, vec, st, ec_adam); break;
    default: s = run_worker<__nv_bfloat16>(h, A, vec, st, ec_adam); break;
  }
  if (s) return s;
  // partials outside the exact range of the fast squares are summed again in double (a scan otherwise)
  const int64_t parts = (int64_t)h->plan.nl * h->plan.wchunks.size();
  s = launch(h, ONEBIT_K_WORKER_SCALE, k_worker_exact,
             grid_for(h, (const void*)k_worker_exact, kThreads, (parts + kThreads - 1) / kThreads), kThreads, st, A);
  if (s) return s;
  const int nt = h->plan.nl * h->plan.T;
  // one partial per range at most: one thread per scale; many short ranges: one warp per scale;
  // otherwise one CTA per scale
  if (h->plan.max_wseg_count <= 1)
    return launch(h, ONEBIT_K_WORKER_SCALE, k_worker_scale_one, (nt + kScaleThreads - 1) / kScaleThreads,
                  kScaleThreads, st, A);
  constexpr int kPerCta = kScaleThreads / 32;
  if (h->plan.max_wseg_count <= kWarpScaleMax)
    return launch(h, ONEBIT_K_WORKER_SCALE, k_worker_scale_warp, (nt + kPerCta - 1) / kPerCta, kScaleThreads, st, A);
  return launch(h, ONEBIT_K_WORKER_SCALE, k_worker_scale, nt, kScaleThreads, st, A);
}

// The server half: K2 over the handle's shards (all, or a rank's own) and the shard scales.
onebit_status_t run_server_half(onebit_adam* h, cudaStream_t st) {
  StepArgs A = base_args(h);
  narrow_to_own_shards(h, &A);
  onebit_status_t s = run_server(h, A, st);
  if (s) return s;
  const int nt = h->plan.n * h->plan.T;
  if (h->plan.max_shard_count <= 1)  // (a rank's own ranges are no longer than the plan's)
    return launch(h, ONEBIT_K_SERVER_SCALE, k_server_scale_one, (nt + kScaleThreads - 1) / kScaleThreads,
                  kScaleThreads, st, A);
  constexpr int kPerCta = kScaleThreads / 32;
  if (h->plan.max_shard_count <= kWarpScaleMax)
    return launch(h, ONEBIT_K_SERVER_SCALE, k_server_scale_warp, (nt + kPerCta - 1) / kPerCta, kScaleThreads, st, A);
  return launch(h, ONEBIT_K_SERVER_SCALE, k_server_scale, nt, kScaleThreads, st, A);
}

// The step's bookkeeping once its last kernel is enqueued.
void finish_step(onebit_adam* h, bool ec_adam) {
  h->compress_steps += 1;
  h->t += 1;
  if (!ec_adam) h->m_dense = false;  // the baseline keeps Adam's own fp32 momentum
  h->werr_zero = false;
  h->serr_zero = false;
}

onebit_status_t do_compress(onebit_adam* h, const void* const* grads, cudaStream_t st, bool ec_adam = false) {
  if (h->phase != (ec_adam ? ONEBIT_PHASE_WARMUP : ONEBIT_PHASE_COMPRESS) || h->xstage) return ONEBIT_ERR_PHASE;
  if (h->plan.world > 1) return ONEBIT_ERR_UNSUPPORTED;  // a rank's step needs the exchange (begin/serve/end)
  onebit_status_t s = run_worker_half(h, grads, st, ec_adam);
  if (s) return s;
  if ((s = run_server_half(h, st))) return s;
  StepArgs A = base_args(h);
  if (ec_adam) {
    const int64_t t = h->t + 1;
    A.bc1 = (float)(1.0 - std::pow((double)h->cfg.beta1, (double)t));
    A.bc2 = (float)(1.0 - std::pow((double)h->cfg.beta2, (double)t));
    auto go = [&](auto k) {
      return launch(h, ONEBIT_K_EC_UPDATE, k, grid_for(h, (const void*)k, kThreads, A.n_chunks), kThreads, st, A);
    };
    const bool bc = h->cfg.bias_correction != 0;
    if (bc) s = h->params_aligned ? go(k_ec_adam_update<true, true>) : go(k_ec_adam_update<true, false>);
    else s = h->params_aligned ? go(k_ec_adam_update<false, true>) : go(k_ec_adam_update<false, false>);
  } else {
    s = run_update(h, A, st);
  }
  if (s) return s;
  finish_step(h, ec_adam);
  return ONEBIT_OK;
}

// ---- the multi-GPU form: the compression step split at the exchange

onebit_status_t run_exchange_copy(onebit_adam* h, int stage, const void* buf, cudaStream_t st) {
  const size_t cnt = h->plan.xr[stage].size();
  if (!cnt) return ONEBIT_OK;
  XArgs X{};
  X.r = h->at<XRange>(h->lay.xr[stage]);
  X.n = (int32_t)cnt;
  const size_t nt = (size_t)h->plan.n * h->plan.T;
  const int cur = (int)(h->compress_steps & 1);
  X.base[0] = h->at<uint32_t>(h->lay.wbits);
  X.base[1] = reinterpret_cast<uint32_t*>(h->at<float>(h->lay.wscale) + cur * nt);
  X.base[2] = h->at<uint32_t>(h->lay.sbits);
  X.base[3] = reinterpret_cast<uint32_t*>(h->at<float>(h->lay.sscale) + cur * nt);
  X.base[4] = const_cast<uint32_t*>(static_cast<const uint32_t*>(buf));
#ifdef ONEBIT_CHECKS
  const Plan& P = h->plan;
  X.words[0] = (int64_t)P.n * P.Wr;
  X.words[1] = (int64_t)nt;
  X.words[2] = P.Wp;
  X.words[3] = (int64_t)nt;
  X.words[4] = stage == 2 ? P.xbcast : (int64_t)P.world * (stage < 2 ? P.xsend : P.xbcast);
  X.status = h->at<unsigned int>(h->lay.status);
#endif
  return launch(h, ONEBIT_K_EXCHANGE, k_exchange_copy, grid_for(h, (const void*)k_exchange_copy, kThreads, X.n),
                kThreads, st, X);
}

onebit_status_t do_begin(onebit_adam* h, const void* const* grads, void* send, cudaStream_t st) {
  if (!h->plan.ranked) return ONEBIT_ERR_UNSUPPORTED;
  if (h->phase != ONEBIT_PHASE_COMPRESS || h->xstage != 0) return ONEBIT_ERR_PHASE;
  if (h->plan.world > 1 && !send) return ONEBIT_ERR_INVALID_ARG;
  onebit_status_t s = run_worker_half(h, grads, st, false);
  if (s) return s;
  if ((s = run_exchange_copy(h, 0, send, st))) return s;
  h->xstage = 1;
  return ONEBIT_OK;
}

onebit_status_t do_serve(onebit_adam* h, const void* recv, void* bcast, cudaStream_t st) {
  if (!h->plan.ranked) return ONEBIT_ERR_UNSUPPORTED;
  if (h->xstage != 1) return ONEBIT_ERR_PHASE;
  if (h->plan.world > 1 && (!recv || !bcast)) return ONEBIT_ERR_INVALID_ARG;
  onebit_status_t s = run_exchange_copy(h, 1, recv, st);
  if (s) return s;
  if ((s = run_server_half(h, st))) return s;
  if ((s = run_exchange_copy(h, 2, bcast, st))) return s;
  h->xstage = 2;
  return ONEBIT_OK;
}

onebit_status_t do_end(onebit_adam* h, const void* gathered, cudaStream_t st) {
  if (!h->plan.ranked) return ONEBIT_ERR_UNSUPPORTED;
  if (h->xstage != 2) return ONEBIT_ERR_PHASE;
  if (h->plan.world > 1 && !gathered) return ONEBIT_ERR_INVALID_ARG;
  onebit_status_t s = run_exchange_copy(h, 3, gathered, st);
  if (s) return s;
  s = run_update(h, base_args(h), st);
  if (s) return s;
  finish_step(h, false);
  h->xstage = 0;
  return ONEBIT_OK;
}

// Export kinds on the padded state, written into the caller's unpadded buffer.
onebit_status_t run_export(onebit_adam* h, int kind, const float* src, const uint32_t* bits, const float* scales,
                           int seg_mul, int shard_mul, float* dst, cudaStream_t st, bool own_shards = false) {
  ExportArgs X{};
  X.chunks = h->at<Chunk>(h->lay.chunks);
  X.n_chunks = (int32_t)h->plan.chunks.size();
  if (own_shards && h->plan.ranked) {  // a rank's server state covers its own shards only
    X.chunks = h->at<Chunk>(h->lay.schunks);
    X.n_chunks = (int32_t)h->plan.schunks.size();
  }
  X.kind = kind;
  X.scale_seg_mul = seg_mul;
  X.scale_shard_mul = shard_mul;
  X.src = src;
  X.bits = bits;
  X.scales = scales;
  X.dst = dst;
#ifdef ONEBIT_CHECKS
  X.Dp = h->plan.Dp;
  X.D = h->plan.D;
  // the callers pass either a whole [T][n] server-scale buffer (shard_mul 1) or one worker's T scales
  X.n_scales = shard_mul ? (int64_t)h->plan.n * h->plan.T : h->plan.T;
  X.status = h->at<unsigned int>(h->lay.status);
#endif
  return launch(h, ONEBIT_K_EXPORT, k_export, grid_for(h, (const void*)k_export, kThreads, X.n_chunks), kThreads, st, X);
}

// scales written by the last compression step
float* last_wscale(onebit_adam* h) {
  const size_t nt = (size_t)h->plan.n * h->plan.T;
  return h->at<float>(h->lay.wscale) + ((h->compress_steps + 1) & 1) * nt;
}
float* last_sscale(onebit_adam* h) {
  const size_t nt = (size_t)h->plan.n * h->plan.T;
  return h->at<float>(h->lay.sscale) + ((h->compress_steps + 1) & 1) * nt;
}

onebit_status_t export_m(onebit_adam* h, float* dst, cudaStream_t st) {
  if (h->m_dense) return run_export(h, kExportCopy, h->at<float>(h->lay.m), nullptr, nullptr, 0, 0, dst, st);
  return run_export(h, kExportBits, nullptr, h->at<uint32_t>(h->lay.sbits), last_sscale(h), h->plan.n, 1, dst, st);
}

// Copy the host gradients of one step into a staging buffer; returns the device pointers and the
// buffer index (to be marked free once the step that reads it is enqueued: release_stage()).
onebit_status_t stage_copy(onebit_adam* h, const void* const* host_grads, cudaStream_t st,
                           std::vector<const void*>* dev, int* idx_out) {
  // copies follow the caller's tensors; bind_grads() cuts them into segments afterwards
  const int n = h->plan.n, T = h->plan.Tu;
  const std::vector<int64_t>& numel = h->plan.unumel;
  const size_t gb = h->cfg.grad_dtype == ONEBIT_F32 ? 4 : 2;
  if (!host_grads) return ONEBIT_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < T; ++k)
      if (numel[k] > 0 && !host_grads[(size_t)i * T + k]) return ONEBIT_ERR_INVALID_ARG;
  if (!h->staging[0]) {
    size_t bytes = 0;
    for (int i = 0; i < n; ++i)
      for (int k = 0; k < T; ++k) bytes += align_up(numel[k] * gb, kAlign);
    for (int b = 0; b < 2; ++b) {
      if (refuse_alloc(h) || cudaMalloc(&h->staging[b], std::max<size_t>(bytes, 1)) != cudaSuccess) {
        cudaGetLastError();
        if (b == 1) cudaFree(h->staging[0]);
        h->staging[0] = h->staging[1] = nullptr;
        return ONEBIT_ERR_NOMEM;
      }
    }
    for (int c = 0; c < kCopyStreams; ++c) {
      ONEBIT_CUDA(h, cudaStreamCreateWithFlags(&h->copy_st[c], cudaStreamNonBlocking));
      ONEBIT_CUDA(h, cudaEventCreateWithFlags(&h->ev_copied[c], cudaEventDisableTiming));
    }
    for (int b = 0; b < 2; ++b) ONEBIT_CUDA(h, cudaEventCreateWithFlags(&h->ev_free[b], cudaEventDisableTiming));
  }
  const int idx = h->stage_next;
  h->stage_next ^= 1;
  uint8_t* base = h->staging[idx];
  for (int c = 0; c < kCopyStreams; ++c)
    if (h->ev_free_recorded[idx]) ONEBIT_CUDA(h, cudaStreamWaitEvent(h->copy_st[c], h->ev_free[idx], 0));
  dev->resize((size_t)n * T);
  size_t off = 0;
  int r = 0;
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < T; ++k) {
      const size_t bytes = numel[k] * gb;
      const size_t q = (size_t)i * T + k;
      (*dev)[q] = base + off;
      const uint8_t* src = static_cast<const uint8_t*>(host_grads[q]);
      for (size_t p = 0; p < bytes; p += kCopyPiece, ++r) {
        const size_t len = std::min(kCopyPiece, bytes - p);
        ONEBIT_CUDA(h, cudaMemcpyAsync(base + off + p, src + p, len, cudaMemcpyHostToDevice,
                                       h->copy_st[r % kCopyStreams]));
      }
      off += align_up(bytes, kAlign);
    }
  for (int c = 0; c < kCopyStreams; ++c) {
    ONEBIT_CUDA(h, cudaEventRecord(h->ev_copied[c], h->copy_st[c]));
    ONEBIT_CUDA(h, cudaStreamWaitEvent(st, h->ev_copied[c], 0));
  }
  *idx_out = idx;
  return ONEBIT_OK;
}

onebit_status_t release_stage(onebit_adam* h, int idx, cudaStream_t st) {
  ONEBIT_CUDA(h, cudaEventRecord(h->ev_free[idx], st));
  h->ev_free_recorded[idx] = true;
  return ONEBIT_OK;
}

// No exception may cross the C ABI: a host allocation that fails (std::bad_alloc) becomes
// ONEBIT_ERR_NOMEM, anything else ONEBIT_ERR_INVALID_ARG.
template <typename F>
onebit_status_t guarded(F&& body) noexcept {
  try {
    return body();
  } catch (const std::bad_alloc&) {
    return ONEBIT_ERR_NOMEM;
  } catch (...) {
    return ONEBIT_ERR_INVALID_ARG;
  }
}

// The plan of a handle: one GPU simulating every worker (rank 0 of 1, ranked = false), or rank `rank`
// of `world` in the multi-GPU form (n a multiple of world; ranked = true, also for world = 1).
onebit_status_t plan_for(const onebit_adam_config_t* cfg, int rank, int world, bool ranked, Plan* P) {
  onebit_status_t s = check_config(cfg);
  if (s) return s;
  if (world < 1 || rank < 0 || rank >= world || cfg->n_workers % world != 0) return ONEBIT_ERR_INVALID_ARG;
  if ((s = make_plan(cfg, P))) return s;
  P->ranked = ranked;
  if (ranked) return make_rank_plan(P, rank, world);
  return ONEBIT_OK;
}

onebit_status_t init_handle(const onebit_adam_config_t* cfg, int rank, int world, bool ranked, float* const* params,
                            void* workspace, size_t workspace_bytes, onebit_stream_t stream, onebit_adam_t** out);

}  // namespace

// =================================================================================== C ABI

extern "C" {

const char* onebit_adam_error_string(onebit_status_t s) {
  switch (s) {
    case ONEBIT_OK: return "ok";
    case ONEBIT_ERR_INVALID_ARG: return "invalid argument";
    case ONEBIT_ERR_PHASE: return "call not legal in the current phase";
    case ONEBIT_ERR_CUDA: return "CUDA runtime error";
    case ONEBIT_ERR_NOMEM: return "out of device memory";
    case ONEBIT_ERR_WORKSPACE: return "workspace too small or misaligned";
    case ONEBIT_ERR_NONFINITE: return "non-finite scale (NaN or Inf in the gradients or state)";
    case ONEBIT_ERR_UNSUPPORTED: return "unsupported request";
    case ONEBIT_ERR_BOUNDS: return "a bounds check of the checked build failed";
  }
  return "unknown status";
}

const char* onebit_adam_last_error(const onebit_adam_t* h) { return h ? h->last_error.c_str() : t_init_error.c_str(); }

onebit_status_t onebit_adam_workspace_size(const onebit_adam_config_t* cfg, size_t* bytes) {
  return onebit_adam_workspace_size_rank(cfg, 0, 1, bytes);
}

onebit_status_t onebit_adam_workspace_size_rank(const onebit_adam_config_t* cfg, int32_t rank, int32_t world,
                                                size_t* bytes) {
  return guarded([&]() -> onebit_status_t {
    if (!bytes) return ONEBIT_ERR_INVALID_ARG;
    Plan P;
    onebit_status_t s = plan_for(cfg, rank, world, world > 1, &P);
    if (s) return s;
    *bytes = make_layout(P).total;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_plan_exchange(const onebit_adam_config_t* cfg, int32_t rank, int32_t world, int64_t* rows,
                                          int64_t cap, int64_t* count, int64_t* send_block, int64_t* bcast_block) {
  return guarded([&]() -> onebit_status_t {
    if (!count || !send_block || !bcast_block || (cap > 0 && !rows)) return ONEBIT_ERR_INVALID_ARG;
    Plan P;
    onebit_status_t s = plan_for(cfg, rank, world, true, &P);
    if (s) return s;
    int64_t q = 0;
    for (int st = 0; st < 4; ++st)
      for (size_t r = 0; r < P.xrows[st].size(); r += 8, ++q)
        if (q < cap) std::copy(P.xrows[st].begin() + r, P.xrows[st].begin() + r + 8, rows + q * 8);
    *count = q;
    *send_block = P.xsend;
    *bcast_block = P.xbcast;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_plan_chunks(const onebit_adam_config_t* cfg, int64_t* rows, int64_t cap, int64_t* count) {
  return guarded([&]() -> onebit_status_t {
    if (!count || (cap > 0 && !rows)) return ONEBIT_ERR_INVALID_ARG;
    onebit_status_t s = check_config(cfg);
    if (s) return s;
    Plan P;
    if ((s = make_plan(cfg, &P))) return s;
    *count = (int64_t)P.chunks.size();
    for (int64_t q = 0; q < std::min<int64_t>(cap, *count); ++q) {
      const Chunk& c = P.chunks[q];
      rows[q * 5 + 0] = c.seg;
      rows[q * 5 + 1] = c.shard;
      rows[q * 5 + 2] = c.start;
      rows[q * 5 + 3] = c.len;
      rows[q * 5 + 4] = c.off;
    }
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_plan_worker_chunks(const onebit_adam_config_t* cfg, int64_t* rows, int64_t cap,
                                               int64_t* count) {
  return guarded([&]() -> onebit_status_t {
    if (!count || (cap > 0 && !rows)) return ONEBIT_ERR_INVALID_ARG;
    onebit_status_t s = check_config(cfg);
    if (s) return s;
    Plan P;
    if ((s = make_plan(cfg, &P))) return s;
    *count = (int64_t)P.wchunks.size();
    for (int64_t q = 0; q < std::min<int64_t>(cap, *count); ++q) {
      const Chunk& c = P.wchunks[q];
      rows[q * 6 + 0] = c.seg;
      rows[q * 6 + 1] = c.shard;
      rows[q * 6 + 2] = c.start;
      rows[q * 6 + 3] = c.len;
      rows[q * 6 + 4] = c.off;
      rows[q * 6 + 5] = c.per;
    }
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_init(const onebit_adam_config_t* cfg, float* const* params, void* workspace,
                                 size_t workspace_bytes, onebit_stream_t stream, onebit_adam_t** out) {
  return init_handle(cfg, 0, 1, false, params, workspace, workspace_bytes, stream, out);
}

onebit_status_t onebit_adam_init_rank(const onebit_adam_config_t* cfg, int32_t rank, int32_t world,
                                      float* const* params, void* workspace, size_t workspace_bytes,
                                      onebit_stream_t stream, onebit_adam_t** out) {
  return init_handle(cfg, rank, world, true, params, workspace, workspace_bytes, stream, out);
}

onebit_status_t onebit_adam_exchange_words(const onebit_adam_t* h, int64_t* send_block, int64_t* bcast_block) {
  if (!h || !send_block || !bcast_block) return ONEBIT_ERR_INVALID_ARG;
  *send_block = h->plan.xsend;
  *bcast_block = h->plan.xbcast;
  return ONEBIT_OK;
}

onebit_status_t onebit_adam_compress_begin(onebit_adam_t* h, const void* const* grads, uint32_t* send,
                                           onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_compress_begin");
    if (!h || !grads) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_begin(h, grads, send, as_stream(stream));
  });
}

onebit_status_t onebit_adam_compress_serve(onebit_adam_t* h, const uint32_t* recv, uint32_t* bcast,
                                           onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_compress_serve");
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_serve(h, recv, bcast, as_stream(stream));
  });
}

onebit_status_t onebit_adam_compress_end(onebit_adam_t* h, const uint32_t* gathered, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_compress_end");
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_end(h, gathered, as_stream(stream));
  });
}

}  // extern "C"

namespace {

onebit_status_t init_handle(const onebit_adam_config_t* cfg, int rank, int world, bool ranked, float* const* params,
                            void* workspace, size_t workspace_bytes, onebit_stream_t stream, onebit_adam_t** out) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_init");
    if (!out || !params) return ONEBIT_ERR_INVALID_ARG;
    *out = nullptr;
    onebit_status_t s = check_config(cfg);
    if (s) return s;
    for (int k = 0; k < cfg->n_tensors; ++k)
      if (!params[k] && cfg->numel[k] > 0) return ONEBIT_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, kAlign)) return ONEBIT_ERR_WORKSPACE;

    Plan plan;  // built before the handle, so that a failure here leaves nothing to release
    if ((s = plan_for(cfg, rank, world, ranked, &plan))) return s;
    onebit_adam* h = new (std::nothrow) onebit_adam();
    if (!h) return ONEBIT_ERR_NOMEM;
    // from here on every exit but success releases the handle (an exception included)
    struct Release {
      onebit_adam* h;
      bool cuda;  // the handle holds CUDA resources: free it through onebit_adam_free
      ~Release() {
        if (h) t_init_error = h->last_error;
        if (h && cuda) onebit_adam_free(h);
        else delete h;
      }
    } release{h, false};
    h->cfg = *cfg;
    h->plan = std::move(plan);
    h->cfg.numel = nullptr;  // the plan keeps its own copy
    h->lay = make_layout(h->plan);
    if (workspace && workspace_bytes < h->lay.total) return ONEBIT_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    release.cuda = true;
    if (cudaGetDevice(&h->device) != cudaSuccess) return cuda_fail(h, cudaGetLastError(), "cudaGetDevice");
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess)
      return cuda_fail(h, cudaGetLastError(), "cudaDeviceGetAttribute");
    if (workspace) {
      h->ws = static_cast<uint8_t*>(workspace);
    } else {
      if (cudaMalloc(&h->ws, h->lay.total) != cudaSuccess) {
        cudaGetLastError();
        h->ws = nullptr;
        return ONEBIT_ERR_NOMEM;
      }
      h->ws_owned = true;
    }
    h->params.resize(h->plan.T);
    for (int k = 0; k < h->plan.Tu; ++k)
      for (int v = h->plan.ufirst[k]; v < h->plan.ufirst[k + 1]; ++v)
        h->params[v] = params[k] ? params[k] + h->plan.voff[v] : nullptr;
    h->params_aligned = true;
    for (float* p : h->params)
      if (!aligned(p, 32)) h->params_aligned = false;
    h->ring.assign(kPtrRing, {});

    // zero every piece of state, then upload the tables
    if (cudaMemsetAsync(h->ws, 0, h->lay.total, st) != cudaSuccess)
      return cuda_fail(h, cudaGetLastError(), "cudaMemsetAsync");
    const Plan& P = h->plan;
    std::vector<uint8_t> tables(h->lay.gptr - h->lay.chunks);
    std::memcpy(tables.data(), P.chunks.data(), P.chunks.size() * sizeof(Chunk));
    std::memcpy(tables.data() + (h->lay.seg_ranges - h->lay.chunks), P.seg_ranges.data(), P.T * sizeof(Range));
    std::memcpy(tables.data() + (h->lay.shard_ranges - h->lay.chunks), P.shard_ranges.data(),
                (size_t)P.T * P.n * sizeof(Range));
    std::memcpy(tables.data() + (h->lay.wchunks - h->lay.chunks), P.wchunks.data(), P.wchunks.size() * sizeof(Chunk));
    std::memcpy(tables.data() + (h->lay.wseg_ranges - h->lay.chunks), P.wseg_ranges.data(), P.T * sizeof(Range));
    std::memcpy(tables.data() + (h->lay.schunks - h->lay.chunks), P.schunks.data(), P.schunks.size() * sizeof(Chunk));
    std::memcpy(tables.data() + (h->lay.sshard_ranges - h->lay.chunks), P.sshard_ranges.data(),
                P.sshard_ranges.size() * sizeof(Range));
    for (int st = 0; st < 4; ++st)
      std::memcpy(tables.data() + (h->lay.xr[st] - h->lay.chunks), P.xr[st].data(), P.xr[st].size() * sizeof(XRange));
    if (cudaMemcpyAsync(h->ws + h->lay.chunks, tables.data(), tables.size(), cudaMemcpyHostToDevice, st) != cudaSuccess)
      return cuda_fail(h, cudaGetLastError(), "upload tables");
    if (cudaMemcpyAsync(h->ws + h->lay.pptr, h->params.data(), P.T * sizeof(float*), cudaMemcpyHostToDevice, st) !=
        cudaSuccess)
      return cuda_fail(h, cudaGetLastError(), "upload params");
    // the pageable sources above are staged before the copies return; wait anyway so that the
    // tables vector may go out of scope with no doubt
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_fail(h, cudaGetLastError(), "init sync");
    release.h = nullptr;  // success: the caller owns the handle
    *out = h;
    return ONEBIT_OK;
  });
}

}  // namespace

extern "C" {

onebit_status_t onebit_adam_free(onebit_adam_t* h) {
  return guarded([&]() -> onebit_status_t {
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    for (auto& tl : h->timed) {
      cudaEventDestroy(tl.start);
      cudaEventDestroy(tl.stop);
    }
    for (auto e : h->event_pool) cudaEventDestroy(e);
    if (h->ws_owned && h->ws) cudaFree(h->ws);
    if (h->vnorm_host) cudaFreeHost(h->vnorm_host);
    if (h->ev_vnorm) cudaEventDestroy(h->ev_vnorm);
    for (int b = 0; b < 2; ++b) {
      if (h->staging[b]) cudaFree(h->staging[b]);
      if (h->ev_free[b]) cudaEventDestroy(h->ev_free[b]);
    }
    for (int c = 0; c < kCopyStreams; ++c) {
      if (h->copy_st[c]) cudaStreamDestroy(h->copy_st[c]);
      if (h->ev_copied[c]) cudaEventDestroy(h->ev_copied[c]);
    }
    delete h;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_warmup_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_warmup_step");
    if (!h || !grads) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_warmup(h, grads, as_stream(stream));
  });
}

onebit_status_t onebit_adam_compress_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_compress_step");
    if (!h || !grads) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_compress(h, grads, as_stream(stream));
  });
}

onebit_status_t onebit_adam_ec_adam_step(onebit_adam_t* h, const void* const* grads, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_ec_adam_step");
    if (!h || !grads) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    return do_compress(h, grads, as_stream(stream), true);
  });
}

onebit_status_t onebit_adam_warmup_step_host(onebit_adam_t* h, const void* const* host_grads, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_warmup_step_host");
    if (!h || !host_grads) return ONEBIT_ERR_INVALID_ARG;
    if (h->phase != ONEBIT_PHASE_WARMUP || h->t >= h->cfg.warmup_steps) return ONEBIT_ERR_PHASE;
    DeviceGuard g(h->device);
    std::vector<const void*> dev;
    int idx = 0;
    onebit_status_t s = stage_copy(h, host_grads, as_stream(stream), &dev, &idx);
    if (s) return s;
    s = do_warmup(h, dev.data(), as_stream(stream));
    const onebit_status_t r = release_stage(h, idx, as_stream(stream));
    return s ? s : r;
  });
}

onebit_status_t onebit_adam_compress_step_host(onebit_adam_t* h, const void* const* host_grads, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_compress_step_host");
    if (!h || !host_grads) return ONEBIT_ERR_INVALID_ARG;
    if (h->phase != ONEBIT_PHASE_COMPRESS || h->xstage) return ONEBIT_ERR_PHASE;
    if (h->plan.world > 1) return ONEBIT_ERR_UNSUPPORTED;  // checked before anything is staged
    DeviceGuard g(h->device);
    std::vector<const void*> dev;
    int idx = 0;
    onebit_status_t s = stage_copy(h, host_grads, as_stream(stream), &dev, &idx);
    if (s) return s;
    s = do_compress(h, dev.data(), as_stream(stream));
    const onebit_status_t r = release_stage(h, idx, as_stream(stream));
    return s ? s : r;
  });
}

onebit_status_t onebit_adam_freeze_variance(onebit_adam_t* h, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_freeze_variance");
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    if (h->phase != ONEBIT_PHASE_WARMUP || h->t < 1) return ONEBIT_ERR_PHASE;
    DeviceGuard g(h->device);
    return do_freeze(h, as_stream(stream));
  });
}

onebit_status_t onebit_adam_get_status(onebit_adam_t* h, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    unsigned int flag = 0;
    cudaStream_t st = as_stream(stream);
    ONEBIT_CUDA(h, cudaMemcpyAsync(&flag, h->ws + h->lay.status, sizeof flag, cudaMemcpyDeviceToHost, st));
    ONEBIT_CUDA(h, cudaStreamSynchronize(st));
    if (flag & kStatusBounds) {  // checked builds only
      static const char* names[ONEBIT_NUM_KERNELS] = {"warmup", "freeze", "worker", "worker_scale", "server",
                                                      "server_scale", "update", "export", "ec_update", "exchange"};
      std::string which;
      for (int k = 0; k < ONEBIT_NUM_KERNELS; ++k)
        if (flag & (1u << (8 + k))) which += (which.empty() ? "" : ", ") + std::string(names[k]);
      h->last_error = "a bounds check skipped work in: " + which;
      return ONEBIT_ERR_BOUNDS;
    }
    if (flag & 2u) {
      h->last_error = "a kernel's wait for its asynchronous copies timed out";
      return ONEBIT_ERR_CUDA;
    }
    return flag ? ONEBIT_ERR_NONFINITE : ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_clear_status(onebit_adam_t* h, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    ONEBIT_CUDA(h, cudaMemsetAsync(h->ws + h->lay.status, 0, sizeof(unsigned int), as_stream(stream)));
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_get_step(const onebit_adam_t* h, int64_t* t, int32_t* phase) {
  if (!h || !t || !phase) return ONEBIT_ERR_INVALID_ARG;
  *t = h->t;
  *phase = h->phase;
  return ONEBIT_OK;
}

onebit_status_t onebit_adam_set_step(onebit_adam_t* h, int64_t t, int32_t phase, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    if (!h || t < 0) return ONEBIT_ERR_INVALID_ARG;
    if (phase == ONEBIT_PHASE_WARMUP) {
      if (t >= h->cfg.warmup_steps) return ONEBIT_ERR_INVALID_ARG;
    } else if (phase == ONEBIT_PHASE_COMPRESS) {
      if (t < 1) return ONEBIT_ERR_INVALID_ARG;
      h->m_dense = true;
      h->werr_zero = true;
      h->serr_zero = true;
    } else {
      return ONEBIT_ERR_INVALID_ARG;
    }
    (void)stream;
    h->t = t;
    h->phase = phase;
    h->xstage = 0;  // a resumed handle starts outside any exchange
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_state_size(const onebit_adam_t* h, int32_t what, size_t* bytes) {
  if (!h || !bytes) return ONEBIT_ERR_INVALID_ARG;
  const Plan& P = h->plan;
  switch (what) {
    case ONEBIT_STATE_M:
    case ONEBIT_STATE_V:
    case ONEBIT_STATE_WORKER_ERROR:
    case ONEBIT_STATE_SERVER_ERROR: *bytes = (size_t)P.D * 4; return ONEBIT_OK;
    case ONEBIT_STATE_WORKER_BITS:
    case ONEBIT_STATE_SERVER_BITS: *bytes = (size_t)P.Wp * 4; return ONEBIT_OK;
    case ONEBIT_STATE_WORKER_SCALES:
    case ONEBIT_STATE_SERVER_SCALES: *bytes = (size_t)P.n * P.T * 4; return ONEBIT_OK;
    default: return ONEBIT_ERR_INVALID_ARG;
  }
}

onebit_status_t onebit_adam_export(onebit_adam_t* h, int32_t what, int32_t worker, void* dst, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_export");
    if (!h || !dst) return ONEBIT_ERR_INVALID_ARG;
    const Plan& P = h->plan;
    const bool per_worker = what == ONEBIT_STATE_WORKER_ERROR || what == ONEBIT_STATE_WORKER_BITS;
    if (per_worker && (worker < 0 || worker >= P.n)) return ONEBIT_ERR_INVALID_ARG;
    // a rank keeps the errors of its own workers only
    if (what == ONEBIT_STATE_WORKER_ERROR && (worker < P.w0 || worker >= P.w0 + P.nl)) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    cudaStream_t st = as_stream(stream);
    float* out = static_cast<float*>(dst);
    switch (what) {
      case ONEBIT_STATE_M: return export_m(h, out, st);
      case ONEBIT_STATE_V: return run_export(h, kExportCopy, h->at<float>(h->lay.v), nullptr, nullptr, 0, 0, out, st);
      case ONEBIT_STATE_WORKER_ERROR:
        if (h->werr_zero)
          return run_export(h, kExportZero, nullptr, nullptr, nullptr, 0, 0, out, st);
        return run_export(h, kExportSignedErr, h->at<float>(h->lay.c) + (size_t)(worker - P.w0) * P.Dp, nullptr,
                          last_wscale(h) + (size_t)worker * P.T, 1, 0, out, st);
      case ONEBIT_STATE_SERVER_ERROR: {
        if (h->serr_zero)
          return run_export(h, kExportZero, nullptr, nullptr, nullptr, 0, 0, out, st);
        if (P.world > 1) {  // other ranks' shards read 0
          const onebit_status_t s = run_export(h, kExportZero, nullptr, nullptr, nullptr, 0, 0, out, st);
          if (s) return s;
        }
        return run_export(h, kExportSignedErr, h->at<float>(h->lay.a), nullptr, last_sscale(h), P.n, 1, out, st,
                          true);
      }
      case ONEBIT_STATE_WORKER_BITS:
        ONEBIT_CUDA(h, cudaMemcpyAsync(dst, h->at<uint32_t>(h->lay.wbits) + (size_t)worker * P.Wr, P.Wp * 4,
                                       cudaMemcpyDeviceToDevice, st));
        return ONEBIT_OK;
      case ONEBIT_STATE_SERVER_BITS:
        ONEBIT_CUDA(h, cudaMemcpyAsync(dst, h->at<uint32_t>(h->lay.sbits), P.Wp * 4, cudaMemcpyDeviceToDevice, st));
        return ONEBIT_OK;
      case ONEBIT_STATE_WORKER_SCALES:
        ONEBIT_CUDA(h, cudaMemcpyAsync(dst, last_wscale(h), (size_t)P.n * P.T * 4, cudaMemcpyDeviceToDevice, st));
        return ONEBIT_OK;
      case ONEBIT_STATE_SERVER_SCALES:
        ONEBIT_CUDA(h, cudaMemcpyAsync(dst, last_sscale(h), (size_t)P.n * P.T * 4, cudaMemcpyDeviceToDevice, st));
        return ONEBIT_OK;
      default: return ONEBIT_ERR_INVALID_ARG;
    }
  });
}

onebit_status_t onebit_adam_import(onebit_adam_t* h, int32_t what, int32_t worker, const void* src, onebit_stream_t stream) {
  return guarded([&]() -> onebit_status_t {
    NvtxRange trace("onebit_adam_import");
    if (!h || !src) return ONEBIT_ERR_INVALID_ARG;
    if (h->xstage) return ONEBIT_ERR_PHASE;  // not in the middle of a split step
    const Plan& P = h->plan;
    DeviceGuard g(h->device);
    cudaStream_t st = as_stream(stream);
    const float* in = static_cast<const float*>(src);
    const size_t nt = (size_t)P.n * P.T;
    onebit_status_t s;
    switch (what) {
      case ONEBIT_STATE_M:
        if ((s = run_export(h, kImportCopy, in, nullptr, nullptr, 0, 0, h->at<float>(h->lay.m), st))) return s;
        h->m_dense = true;
        return ONEBIT_OK;
      case ONEBIT_STATE_V:
        return run_export(h, kImportCopy, in, nullptr, nullptr, 0, 0, h->at<float>(h->lay.v), st);
      case ONEBIT_STATE_WORKER_ERROR: {
        if (worker < P.w0 || worker >= P.w0 + P.nl) return ONEBIT_ERR_INVALID_ARG;  // this rank's workers only
        float* ws_prev = last_wscale(h);  // what the next step reads as the previous scales
        if (h->werr_zero) {
          ONEBIT_CUDA(h, cudaMemsetAsync(h->at<float>(h->lay.c), 0, (size_t)P.nl * P.Dp * 4, st));
          ONEBIT_CUDA(h, cudaMemsetAsync(ws_prev, 0, nt * 4, st));
          h->werr_zero = false;
        }
        // store delta as c with a zero scale: the next step rebuilds c - 0*sign(c) = delta exactly
        if ((s = run_export(h, kImportCopy, in, nullptr, nullptr, 0, 0,
                            h->at<float>(h->lay.c) + (size_t)(worker - P.w0) * P.Dp, st)))
          return s;
        ONEBIT_CUDA(h, cudaMemsetAsync(ws_prev + (size_t)worker * P.T, 0, (size_t)P.T * 4, st));
        return ONEBIT_OK;
      }
      case ONEBIT_STATE_SERVER_ERROR: {
        if (!h->m_dense) {  // m is carried by the server scales about to be zeroed: materialise it
          if ((s = export_m(h, h->at<float>(h->lay.m), st))) return s;
          h->m_dense = true;
        }
        // store eps as a with a zero scale: the next step rebuilds a - 0*sign(a) = eps exactly (a rank
        // keeps the errors of its own shards only)
        if ((s = run_export(h, kImportCopy, in, nullptr, nullptr, 0, 0, h->at<float>(h->lay.a), st, true))) return s;
        ONEBIT_CUDA(h, cudaMemsetAsync(last_sscale(h), 0, nt * 4, st));
        h->serr_zero = false;
        return ONEBIT_OK;
      }
      default: return ONEBIT_ERR_INVALID_ARG;
    }
  });
}

onebit_status_t onebit_adam_comm_bytes(const onebit_adam_t* h, uint64_t* compressed, uint64_t* fp32_bytes) {
  if (!h || !compressed || !fp32_bytes) return ONEBIT_ERR_INVALID_ARG;
  uint64_t c = 0, f = 0;
  for (int64_t L : h->plan.numel) {
    c += (uint64_t)((L + 31) / 32) * 4 + 4;
    f += (uint64_t)L * 4;
  }
  *compressed = c;
  *fp32_bytes = f;
  return ONEBIT_OK;
}

onebit_status_t onebit_adam_set_timing(onebit_adam_t* h, int32_t enable) {
  return guarded([&]() -> onebit_status_t {
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    h->timing = enable != 0;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_kernel_times(onebit_adam_t* h, double* ms, int64_t* launches) {
  return guarded([&]() -> onebit_status_t {
    if (!h || !ms || !launches) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    for (int k = 0; k < ONEBIT_NUM_KERNELS; ++k) {
      ms[k] = 0.0;
      launches[k] = 0;
    }
    onebit_status_t rc = ONEBIT_OK;
    for (auto& tl : h->timed) {
      float t = 0.0f;
      if (cudaEventSynchronize(tl.stop) != cudaSuccess || cudaEventElapsedTime(&t, tl.start, tl.stop) != cudaSuccess)
        rc = cuda_fail(h, cudaGetLastError(), "kernel timing");
      ms[tl.kernel] += t;
      launches[tl.kernel] += 1;
      h->event_pool.push_back(tl.start);
      h->event_pool.push_back(tl.stop);
    }
    h->timed.clear();
    return rc;
  });
}

onebit_status_t onebit_adam_set_variance_monitor(onebit_adam_t* h, int32_t enable) {
  return guarded([&]() -> onebit_status_t {
    if (!h) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (enable) {
      const onebit_status_t s = ensure_vnorm_slot(h);
      if (s) return s;
    }
    h->vmon = enable != 0;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_set_auto_freeze(onebit_adam_t* h, double tol) {
  return guarded([&]() -> onebit_status_t {
    if (!h || !std::isfinite(tol) || tol < 0.0) return ONEBIT_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (tol > 0.0) {
      const onebit_status_t s = ensure_vnorm_slot(h);
      if (s) return s;
    }
    h->auto_tol = tol;
    h->auto_have_prev = false;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_variance_norm(onebit_adam_t* h, double* norm, int64_t* step) {
  return guarded([&]() -> onebit_status_t {
    if (!h || !norm || !step) return ONEBIT_ERR_INVALID_ARG;
    if (h->vnorm_step == 0) return ONEBIT_ERR_PHASE;  // no monitored warm-up step yet
    DeviceGuard g(h->device);
    ONEBIT_CUDA(h, cudaEventSynchronize(h->ev_vnorm));
    *norm = *h->vnorm_host;
    *step = h->vnorm_step;
    return ONEBIT_OK;
  });
}

onebit_status_t onebit_adam_set_fault_injection(onebit_adam_t* h, int32_t kind, int64_t value) {
  if (!h) return ONEBIT_ERR_INVALID_ARG;
  switch (kind) {
    case ONEBIT_FAULT_NONE:
      h->stall_tx = 0;
      h->fail_allocs = 0;
      h->check_margin = 0;
      return ONEBIT_OK;
    case ONEBIT_FAULT_STALL_COPIES:
      if (value < 1 || value > (1 << 20)) return ONEBIT_ERR_INVALID_ARG;
      h->stall_tx = (uint32_t)value;
      return ONEBIT_OK;
    case ONEBIT_FAULT_FAIL_ALLOC:
      if (value < 1 || value > 1000) return ONEBIT_ERR_INVALID_ARG;
      h->fail_allocs = (int)value;
      return ONEBIT_OK;
    case ONEBIT_FAULT_TIGHTEN_BOUNDS:
#ifdef ONEBIT_CHECKS
      if (value < 1 || value % 32 || value > h->plan.Dp) return ONEBIT_ERR_INVALID_ARG;
      h->check_margin = value;
      return ONEBIT_OK;
#else
      return ONEBIT_ERR_UNSUPPORTED;  // a normal build has no bounds checks to tighten
#endif
    default: return ONEBIT_ERR_INVALID_ARG;
  }
}

onebit_status_t onebit_adam_set_lr(onebit_adam_t* h, float lr) {
  if (!h || !std::isfinite(lr)) return ONEBIT_ERR_INVALID_ARG;
  h->cfg.lr = lr;
  return ONEBIT_OK;
}

onebit_status_t onebit_adam_set_max_ctas(onebit_adam_t* h, int32_t max_ctas) {
  if (!h || max_ctas < 0) return ONEBIT_ERR_INVALID_ARG;
  h->max_ctas = max_ctas;
  return ONEBIT_OK;
}

onebit_status_t onebit_adam_launch_count(const onebit_adam_t* h, int64_t* launches) {
  if (!h || !launches) return ONEBIT_ERR_INVALID_ARG;
  *launches = h->launches;
  return ONEBIT_OK;
}

}  // extern "C"
