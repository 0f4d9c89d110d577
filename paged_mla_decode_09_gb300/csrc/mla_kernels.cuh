// Device code of the paged MLA decode: constants, shared-memory layout,
// schedule (K0), split-KV attention (K1), log-sum-exp combine (K2), the TMA
// gather test hook and the bounded-wait self-test.
//
// Method: TokenSpeed code audit (mlqm.cn/news/403565), 完整技术清单 > MLA —
// one latent row per token serving as key (576) and value (512), two-stage
// split-KV decode with fp32 partials merged by log-sum-exp.  Tiling and the
// online softmax follow the FlashAttention article of the guijiagi.com
// "推理优化" tag page (same result as plain attention).
//
// GB300 design (one row block = up to 128 query rows = heads x drafts):
//   * a thread-block cluster is one CTA PAIR; with G row blocks, G clusters
//     compute the same slice of pages, one row block each;
//   * the S CTA keeps the row block's absorbed queries in TMEM and computes
//     S = Q K^T per 64-token page with tcgen05 (A from TMEM, B = the page,
//     K-major), then the online softmax (one thread per row) and writes the
//     probabilities P straight into the O CTA's shared memory (DSMEM);
//   * the O CTA keeps the 128 x 512 fp32 output accumulator in TMEM (all
//     512 columns) and computes O += P V with V = the same page read through
//     an MN-major descriptor, applying lazy output rescales;
//   * pages arrive by TMA (128-byte swizzled boxes of 64 tokens) through the
//     page table; shared prefix pages are just the same ids, read in place;
//   * the cluster walks a contiguous, page-balanced slice of all requests'
//     pages; requests cut by a slice boundary write fp32 partials that the
//     combine kernel merges by log-sum-exp.
//
// Every barrier below is used so that its completer can never run two phases
// ahead of a waiter (parity waits would then miss a phase).  Where a chain
// of barriers does not already guarantee that, the barrier is split per
// P slot (p_full, p_empty).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "mla_decode.h"
#include "sm100_ptx.cuh"

namespace mla {

constexpr int kPage = 64;
constexpr int kDL = 512;
constexpr int kDR = 64;
constexpr int kRows = 128;     // rows per row block = M of every MMA
// 12 warps: 0 TMA, 1 and 3 MMA, 2 TMEM alloc, 4-11 row warps in two groups
// of four (warps 4-7 and 8-11; each group has one thread per query row).  In
// the S CTA the groups take alternate pages (one group's P transfer overlaps
// the other's softmax); in the O CTA they take one half each of the 512
// output columns.
constexpr int kThreads = 384;
constexpr int kRowThreads = 256;
constexpr int kRowWarps = 8;  // row-warp barriers take one arrival per warp (lane 0, after __syncwarp)
constexpr int kNS = 3;         // S accumulators in TMEM (S CTA)
constexpr uint32_t kSCol0 = 320;  // TMEM column of S buffer 0 (queries use 0..287)
constexpr int kCtrlBytes = 512;
// Schedule weight of starting a request piece, in pages: a cluster pays a
// fixed cost per piece it starts (queries into TMEM, pipeline refill,
// epilogue).  Measured on GB300 (per-cluster times regressed on the pages
// and pieces of their slices, and sweeps): about 6 pages' time for a block
// of 128 rows, 3-4 for one of at most 64 rows (half the queries to load and
// half the output to store).  With e4m3, 6 was best when the scale pre-pass
// prepares the query terms; when the attention kernel splits the rows
// itself the step was flat within 0.3 % from 8 to 14, and the same 6 keeps
// both query paths on one schedule (bit-identical results).
__host__ __device__ constexpr int unit_cost_pages(bool f8, int block_rows) {
  return f8 ? 6 : (block_rows <= 64 ? 4 : 6);
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Lazy output rescale: O is rescaled only when a row's running max grows by
// more than the threshold (log2 units).  P is computed relative to the stale
// max, times 2^shift, so that it never exceeds 2^(threshold + shift) (bf16:
// threshold 8, no shift).  For e4m3, threshold 6 and shift 2 keep P at most
// 2^8 (e4m3's largest finite value is 448) while the bulk of the
// probability mass stays out of its subnormals (with no shift, the many
// small P of a long row lose enough in the hi + lo split to reach 0.8 of
// the parity tolerance in simulation; with shift 2, 0.11); an integral shift
// keeps the P of a row's max key (2^shift) exact.
// Every page on which one of the block's rows crosses the threshold stalls
// PV for an O rescale (measured: ~1.3 us of PV time per such page): over a
// long sequence of Gaussian-like scores one of 128 rows crosses 3 on most
// pages, 5 on about one page in eight, 6 on fewer.  The shift cancels in
// out = O / l and is removed from the lse.
template <bool kF8>
struct SoftmaxCfg {
  static constexpr float kThreshold = kF8 ? 6.0f : 8.0f;
  static constexpr float kShift = kF8 ? 2.0f : 0.0f;
  static_assert(kThreshold + kShift <= 8.f, "P must stay below e4m3's largest finite value");
};
constexpr float kMinusBig = -1.0e30f;      // running-max sentinel (finite, so exp2 never sees inf - inf)

template <bool kF8>
struct Cfg {
  static constexpr int kEsz = kF8 ? 1 : 2;
  static constexpr int kBox = 8192;                     // one TMA box: 64 tokens x 128 bytes
  static constexpr int kNBoxLat = kF8 ? 4 : 8;          // boxes holding c_kv
  static constexpr int kPeBytes = kF8 ? 4096 : 8192;    // box holding k_pe
  static constexpr int kSlotS = kNBoxLat * kBox + kPeBytes;
  static constexpr int kSlotO = kNBoxLat * kBox;
  static constexpr int kNStS = kF8 ? 6 : 3;
  static constexpr int kNStO = kF8 ? 5 : 3;
  // One copy per page (measured on GB300: three 24 KB copies per page
  // instead of one 72 KB copy raise the copy latency about threefold).
  static constexpr int kBoxesPartS = kF8 ? 4 : 9;   // boxes of the c_kv / whole-row map per copy
  static constexpr int kBoxesPartO = kF8 ? 4 : 8;
  static constexpr int kPBytes = kRows * kPage * kEsz;  // one P tile
  static constexpr int kPRow = kPage * kEsz;            // bytes of one P row (128 or 64)
  static constexpr int kKStepsPe = kF8 ? 2 : 4;         // 32-byte K steps in the k_pe box
  static constexpr uint32_t kPeSwz = kF8 ? kSwizzle64B : kSwizzle128B;
  static constexpr uint32_t kPeSbo = kF8 ? 512 : 1024;
  // P tile: K-major without swizzle.  Core matrices of 8 rows x 16 bytes
  // (8 keys bf16, 16 keys e4m3); the 16-byte chunk c of row r sits at
  // (r / 8) * kPSbo + c * kPLbo + (r % 8) * 16, so chunk c of 8 consecutive
  // rows is 128 contiguous bytes and a warp storing chunk c of its 32 rows
  // into the O CTA writes four whole 128-byte lines (one row per thread and
  // a swizzled tile would touch 32 lines with 16 bytes each).
  static constexpr uint32_t kPSwz = kSwizzleNone;
  static constexpr uint32_t kPLbo = 128;                // next core matrix along K
  static constexpr uint32_t kPSbo = kF8 ? 512 : 1024;   // next 8-row group
  static constexpr int kPChunks = kF8 ? 4 : 8;          // 16-byte chunks per P row
  // e4m3 P is sent as two terms hi + lo (hi = e4m3(p), lo = e4m3(p - hi)),
  // two 8 KB tiles of one slot, both multiplied by the same V page: one
  // e4m3 term alone (3 mantissa bits) moves a row's weights by a few
  // percent when it sees only a handful of keys
  static constexpr int kPTerms = kF8 ? 2 : 1;
  static constexpr uint32_t kPTermBytes = kRows * kPage;  // e4m3: 8 KB
  static constexpr int kPvKSteps = kF8 ? 2 : 4;         // K = 64 tokens in steps of 32 (e4m3) / 16 (bf16)
  static constexpr int kVKStepBytes = kF8 ? 4096 : 2048;
  static constexpr int kVBoxesHalf = kF8 ? 2 : 4;       // boxes covering 256 output columns
  // e4m3 queries are stored as two terms hi + lo sharing one per-row scale
  // (hi = e4m3(q/s), lo = e4m3(q/s - hi)); both multiply the same K page and
  // accumulate into the same S, giving about bf16 precision for q.
  static constexpr int kQSplit = kF8 ? 2 : 1;
  static constexpr uint32_t kQLoCol = 144;              // TMEM column of the lo term
  static constexpr uint32_t kIdescQK = make_idesc(kF8, 128, 64, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(kF8, 128, 256, false, true);
  static constexpr int kMlOff = kNStS * kSlotS;          // S CTA: (m0, l0, m1, l1)[128], one pair per group
  // S CTA: the row references of the last 4 pages [4][128] (page tag, value)
  static constexpr int kPubOff = kMlOff + 4 * kRows * 4;
  static constexpr int kDataS = kPubOff + 4 * kRows * 8;
  // O CTA: P slots first (a slot's padding rows read on into what follows,
  // which must be shared memory of this CTA), then the c_kv ring, then the
  // row references that come with each P
  static constexpr int kPOff = 0;
  static constexpr int kPRegion = kF8 ? 3 * 16384 : 4 * 8192;
  static constexpr int kRingOffO = kPOff + kPRegion;
  static constexpr int kRefOff = kRingOffO + kNStO * kSlotO;
  static constexpr int kRefBytes = (kF8 ? 3 : 2) * kRows * 4;
  static constexpr int kFlagOff = kRefOff + kRefBytes;  // per P slot: one word per softmax warp (rows that rose)
  static constexpr int kDataO = kFlagOff + 4 * 16;
  static constexpr int kData = kDataS > kDataO ? kDataS : kDataO;
  // dynamic smem = alignment slack + 1024-aligned data + control block
  static constexpr int kSmem = 1024 + kData + kCtrlBytes;
  // bytes the S CTA sends per page: per real query row its P row and O
  // scale factor, and one flag word per softmax warp
  static constexpr uint32_t kPTxRow = kPRow * kPTerms + 4;
  static constexpr uint32_t kPTxFlags = 4 * 4;
  static_assert(kSmem <= 232448, "shared memory budget");
};

// P slots of a row block in the O CTA.  bf16: a P row is 128 bytes; with at
// most 64 real rows a slot needs only 8 KB (the MMA's rows 64-127 read the
// next 8 KB, whose results land in O rows that are never stored), so the
// 32 KB region holds 4 slots, else 2 of 16 KB.  e4m3: 3 slots of 16 KB,
// each the hi and the lo tile (8 KB each) of one page.
struct PSlots {
  int n;            // slots
  uint32_t stride;  // bytes from one slot to the next
  int arows;        // reference entries per slot
  __device__ PSlots(bool f8, int rows_real) {
    if (f8) {
      n = 3; stride = 16384; arows = kRows;  // hi and lo tiles
    } else if (rows_real <= 64) {
      n = 4; stride = 8192; arows = 64;
    } else {
      n = 2; stride = 16384; arows = kRows;
    }
  }
};
constexpr int kMaxPSlots = 4;

struct __align__(8) Ctrl {
  uint64_t kv_full[6];   // one per ring slot
  uint64_t kv_empty[6];
  uint64_t s_full[kNS];
  uint64_t s_empty[kNS];
  uint64_t q_full;  // queries of the unit loaded into TMEM
  uint64_t p_full[kMaxPSlots];
  uint64_t p_empty[kMaxPSlots];
  uint64_t o_full;
  uint64_t o_empty;
  uint64_t resc_req;   // O CTA: page resc_page needs O rescaled (waiter -> correction warps)
  uint64_t resc_done;  // O CTA: the correction warps rescaled O
  uint64_t ml_full;
  uint64_t ml_empty;
  uint64_t pv_ready;  // O CTA: page j is ready for PV (waiter warp -> MMA warp)
  uint64_t pv_taken;  // O CTA: the MMA warp took page j (keeps the waiter one page ahead at most)
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t resc_page;
  int abort;
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block");

struct Params {
  const uint8_t* q_nope;   // bf16
  const uint8_t* q_pe;     // bf16
  const int32_t* page_table;
  const int32_t* seq_lens;
  uint8_t* out;            // bf16
  float* lse;
  float* o_part;           // [2C][G][128][512]
  float* lse_part;         // [2C][G][128]
  int32_t* status;         // [4]: status bits, timeout diagnostics
  int32_t* prefix;         // [B+1] page prefix sums
  int32_t* cinfo;          // [C][3] = slice start, slice end, first request
  int32_t* rrange;         // [B][2] = first and last cluster whose slice meets the request
  int32_t* splits;         // [8] count, then [min(B, C)][8] = (request, pieces, partial slots of the first 6)
                           // for each request cut into pieces (any order)
  float* qscale;           // [B * R] e4m3 query scales (e4m3 cache only)
  // e4m3 cache: [B * R][1152] each query row's e4m3 terms, hi (576 bytes)
  // then lo, written by the scale pre-pass and copied into the S CTA's ring
  // like the bf16 query rows; null: the attention kernel splits the rows
  // itself (the allocation-free entry point when they do not fit its scratch)
  uint8_t* qterms;
  int32_t B, H, Q, R, G, C;
  int32_t num_pages, max_pages, pt_stride;
  int32_t unit_cost;       // schedule weight of a request piece, in pages
  int32_t out_f32;         // out is fp32 [B][Q][H][512] instead of bf16 (internal: the cascade's passes)
  int32_t len_offset;      // request b's length is seq_lens[b] - len_offset (internal: the cascade's suffix pass)
  int32_t len_fixed;       // > 0: every request's length, seq_lens unread (internal: the cascade's prefix pass)
  // internal, the top-k decode over packed pick lists (null otherwise): the
  // gather's status bits, one word per (list, chunk of picks), are OR-ed into
  // the status word by the schedule; a list without a valid pick gets the lse
  // of an empty key set, -inf, from the combine's block 0
  const int32_t* topk_bits;
  const int32_t* topk_empty;  // [B]
  int32_t topk_nchunk;
  float scale, kv_scale;
  uint64_t timeout_ns;
};

// Optional event trace (built only with -DMLA_TRACE): global-timer stamps
// of each pipeline event per page for one cluster, for latency analysis, and
// of each cluster's start and end and the kernels' entries and exits.  With
// -DMLA_TRACE_NO_PAGES as well, only the latter (a few stamps per cluster:
// timings close to those of the normal build).
#ifdef MLA_TRACE
__device__ uint64_t g_mla_trace[2][16][1024];
// per cluster: [0] start, [1] S producer done, [2] O epilogue of the last unit done
__device__ uint64_t g_mla_cluster_times[1024][4];
__device__ int g_mla_trace_cid;  // the cluster whose events are stamped
// [0] schedule entry, [1] schedule exit, [2] first combine block entry
// (after its wait), [3] last combine block exit, [4] first attention CTA
// entry, [5] first attention CTA past its wait
__device__ unsigned long long g_mla_kernel_times[8];
// combine blocks: [block][0] past the wait, [1] record loaded, [2] partials
// loaded, [3] stored (first warp of the block)
__device__ unsigned long long g_mla_combine_times[4096][4];
#define MLA_COMBINE_STAMP(k)                                                  \
  do {                                                                        \
    const unsigned bid = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z); \
    if (threadIdx.x == 0 && bid < 4096) g_mla_combine_times[bid][(k)] = globaltimer_ns(); \
  } while (0)
#else
#define MLA_COMBINE_STAMP(k) \
  do {                       \
  } while (0)
#endif
#if defined(MLA_TRACE) && !defined(MLA_TRACE_NO_PAGES)
#define MLA_TRACE_POINT(role, ev, j)                                                                     \
  do {                                                                                                   \
    if (cluster_id_x() == static_cast<uint32_t>(g_mla_trace_cid) && cluster_ctarank() < 2 && (j) < 1024) \
      g_mla_trace[(role)][(ev)][(j)] = globaltimer_ns();                                                 \
  } while (0)
#else
#define MLA_TRACE_POINT(role, ev, j) \
  do {                               \
  } while (0)
#endif

// Request b's length as this call sees it (see len_offset, len_fixed).
__device__ __forceinline__ int req_len(const int32_t* seq_lens, int b, int len_offset, int len_fixed) {
  return len_fixed > 0 ? len_fixed : seq_lens[b] - len_offset;
}

__device__ __forceinline__ int clamp_len(int L, int max_pages) {
  return L < 0 ? 0 : (L > max_pages * kPage ? max_pages * kPage : L);
}

// ---------------------------------------------------------------- K0
// Page prefix sums over requests and each cluster's page slice
// [T*c/C, T*(c+1)/C) with the request holding its first page.
constexpr int kSchedSmemB = 4096;     // requests whose prefix sums the schedule keeps in shared memory
constexpr int kSchedSmemC = 512;      // clusters whose slices it keeps there
// What cutting requests into pieces costs beyond the pieces' start-up, in
// pages: the combine kernel's launch and wait, and the fp32 partials that
// each piece writes and the combine reads back (a 128-row partial is 256 KB,
// about three and a half bf16 pages, each way).
constexpr int kSplitPenaltyPages = 8;

__global__ void __launch_bounds__(1024) mla_schedule_kernel(Params p) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  // the searches below run on shared-memory copies (a binary search over
  // global memory is a chain of dependent loads); larger batches read the
  // global arrays
  __shared__ int32_t sp[kSchedSmemB + 1];
  __shared__ int32_t cs[kSchedSmemC], ce[kSchedSmemC], cf[kSchedSmemC];
  __shared__ int32_t cnz[kSchedSmemC + 1];  // non-empty slices among clusters [0, c)
  __shared__ int32_t nsplit;
  __shared__ int32_t maxnp;
  // 1024 threads, or 256 for a batch and a cluster count below 256 (fewer
  // warps to gather at each barrier)
  const int nt = static_cast<int>(blockDim.x), nwarps = nt >> 5;
  const bool sp_ok = p.B <= kSchedSmemB;
  const bool c_ok = p.C <= kSchedSmemC && p.C < nt;  // one cluster per thread
  griddep_launch_dependents();  // the next kernels wait for this one before reading its output
  const int tid = threadIdx.x;
#ifdef MLA_TRACE
  if (tid == 0) g_mla_kernel_times[0] = globaltimer_ns();
#endif
  if (tid == 0) {
    carry = 0;
    nsplit = 0;
    maxnp = 0;
  }
  // the top-k gather's status bits (it ended before this kernel began):
  // loaded now, OR-ed into the status word at the end, so that the loads
  // overlap the rest of the schedule
  int topk_bits = 0;
  if (p.topk_bits)
    for (int64_t k = tid; k < static_cast<int64_t>(p.B) * p.topk_nchunk; k += nt) topk_bits |= p.topk_bits[k];
  // the status words start each call at zero: nothing writes them before
  // this kernel, and every later writer waits for it (griddep_wait)
  if (tid < 4) p.status[tid] = 0;
  __syncthreads();
  for (int base = 0; base < p.B; base += nt) {
    const int b = base + tid;
    int np = 0;
    if (b < p.B) {
      const int L = req_len(p.seq_lens, b, p.len_offset, p.len_fixed);
      if (L < p.Q || L > p.max_pages * kPage) atomicOr(p.status, MLA_DEV_BAD_SEQ_LEN);
      np = (clamp_len(L, p.max_pages) + kPage - 1) / kPage;
    }
    int m = np;  // the longest request
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0 && m > 0) atomicMax(&maxnp, m);
    int v = np;  // block-wide inclusive scan
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, v, o);
      if ((tid & 31) >= o) v += t;
    }
    if ((tid & 31) == 31) warp_tot[tid >> 5] = v;
    __syncthreads();
    if (tid < 32) {
      int w = tid < nwarps ? warp_tot[tid] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, w, o);
        if (tid >= o) w += t;
      }
      warp_tot[tid] = w;
    }
    __syncthreads();
    const int incl = v + ((tid >> 5) ? warp_tot[(tid >> 5) - 1] : 0) + carry;
    if (b < p.B) {
      p.prefix[b + 1] = incl;
      if (sp_ok) sp[b + 1] = incl;
    }
    __syncthreads();
    if (tid == nt - 1) carry = incl;
    __syncthreads();
  }
  if (tid == 0) {
    p.prefix[0] = 0;
    sp[0] = 0;
  }
  __syncthreads();
#ifdef MLA_TRACE
  if (tid == 0) g_mla_kernel_times[6] = globaltimer_ns();  // lengths loaded and scanned
#endif
  const int32_t* pre = sp_ok ? sp : p.prefix;
  // Cluster slices are cut in a weighted order: request b occupies
  // p.unit_cost start-up units and then its pages, so clusters whose
  // slice starts many pieces get fewer pages.  A weighted position maps to
  // the page at that point (start-up units map to the request's first page).
  const int64_t T = pre[p.B];
  const int64_t W = T + static_cast<int64_t>(p.unit_cost) * p.B;
  auto page_at = [&](int64_t x) -> int {
    int lo = 0, hi = p.B - 1;  // last request b with prefix[b] + unit_cost * b <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] + static_cast<int64_t>(p.unit_cost) * mid <= x) lo = mid; else hi = mid - 1;
    }
    const int64_t np = pre[lo + 1] - pre[lo];
    int64_t off = x - pre[lo] - static_cast<int64_t>(p.unit_cost) * lo - p.unit_cost;
    off = off < 0 ? 0 : (off > np ? np : off);
    return static_cast<int>(pre[lo] + off);
  };
  // A batch of no more requests than slices whose longest request costs
  // about an even slice gets one request per slice instead: nothing is cut
  // into pieces, so no partials are written and nothing is merged.
  const bool whole = p.B <= p.C && (static_cast<int64_t>(maxnp) + p.unit_cost) * p.C <=
                                       W + static_cast<int64_t>(kSplitPenaltyPages) * p.C;
  // weighted cut positions W * c / C in 32-bit arithmetic when they fit
  const bool cut32 = W * p.C < (static_cast<int64_t>(1) << 31);
  auto cut = [&](int c) -> int64_t {
    return cut32 ? static_cast<int64_t>(static_cast<uint32_t>(W) * static_cast<uint32_t>(c) /
                                        static_cast<uint32_t>(p.C))
                 : W * c / p.C;
  };
  for (int c = tid; c < p.C; c += nt) {
    int s, e, lo;
    if (whole) {  // slice c = request c; the slices past the batch are empty
      s = c < p.B ? pre[c] : static_cast<int>(T);
      e = c < p.B ? pre[c + 1] : static_cast<int>(T);
      lo = c < p.B ? c : p.B - 1;
    } else {
      s = page_at(cut(c));
      e = page_at(cut(c + 1));
      lo = 0;
      int hi = p.B - 1;  // last request b with prefix[b] <= s
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= s) lo = mid; else hi = mid - 1;
      }
    }
    p.cinfo[3 * c + 0] = s;
    p.cinfo[3 * c + 1] = e;
    p.cinfo[3 * c + 2] = lo;
    if (c_ok) {
      cs[c] = s;
      ce[c] = e;
      cf[c] = lo;
    }
  }
  // C <= 512 and below the thread count: thread c wrote cluster c's slice;
  // a ballot per warp of the non-empty ones, then each cluster's count of
  // those before it
  const unsigned m = c_ok ? __ballot_sync(0xffffffffu, tid < p.C && cs[tid] != ce[tid]) : 0u;
  if (c_ok && (tid & 31) == 0) warp_tot[tid >> 5] = __popc(m);
  __syncthreads();
  if (c_ok) {
    if (tid <= p.C) {
      int k = __popc(m & ((1u << (tid & 31)) - 1u));
      for (int w = 0; w < (tid >> 5); ++w) k += warp_tot[w];
      cnz[tid] = k;
    }
    __syncthreads();
  }
#ifdef MLA_TRACE
  if (tid == 0) g_mla_kernel_times[7] = globaltimer_ns();  // cluster slices written
#endif
  // per request, the clusters whose slice [s, e) meets its pages
  // [prefix[b], prefix[b+1]): from the first with e > prefix[b] to the last
  // with s < prefix[b+1] (both bounds are non-decreasing in the cluster
  // index); the combine merges the pieces of requests with more than one
  for (int b = tid; b < p.B; b += nt) {
    const int pb0 = pre[b], pb1 = pre[b + 1];
    int lo = 0, hi = p.C - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if ((c_ok ? ce[mid] : p.cinfo[3 * mid + 1]) > pb0) hi = mid; else lo = mid + 1;
    }
    const int clo = lo;
    lo = 0;
    hi = p.C - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((c_ok ? cs[mid] : p.cinfo[3 * mid]) < pb1) lo = mid; else hi = mid - 1;
    }
    p.rrange[2 * b] = pb1 > pb0 ? clo : 0;
    p.rrange[2 * b + 1] = pb1 > pb0 ? lo : 0;
    // the request's pieces in cluster order (empty slices hold none) and
    // their partial slots: 2c for the piece that starts cluster c's slice,
    // 2c + 1 for a later one.  A request cut into pieces gets an entry of
    // the combine's list: (b, pieces, the first 6 slots).
    int n = 0;
    int32_t rec[8] = {b, 0, 0, 0, 0, 0, 0, 0};
    if (pb1 > pb0 && lo > clo) {
      auto empty = [&](int c) { return c_ok ? cs[c] == ce[c] : p.cinfo[3 * c] == p.cinfo[3 * c + 1]; };
      if (c_ok) {
        n = cnz[lo + 1] - cnz[clo];
      } else {
        for (int c = clo; c <= lo; ++c) n += empty(c) ? 0 : 1;
      }
      int c = clo;
#pragma unroll
      for (int k = 0; k < 6; ++k) {  // unrolled: rec is indexed statically (registers)
        while (c <= lo && empty(c)) ++c;
        if (c <= lo) {
          rec[2 + k] = 2 * c + (b != (c_ok ? cf[c] : p.cinfo[3 * c + 2]) ? 1 : 0);
          ++c;
        }
      }
    }
    rec[1] = n;
    if (n > 1) {  // at most min(B, C - 1) requests
      int4* dst = reinterpret_cast<int4*>(p.splits + 8 * (1 + static_cast<int64_t>(atomicAdd(&nsplit, 1))));
      dst[0] = make_int4(rec[0], rec[1], rec[2], rec[3]);
      dst[1] = make_int4(rec[4], rec[5], rec[6], rec[7]);
    }
  }
  __syncthreads();
  if (tid == 0) p.splits[0] = nsplit;
  if (p.topk_bits) {
    topk_bits = __reduce_or_sync(0xffffffffu, topk_bits);
    if ((tid & 31) == 0 && topk_bits) atomicOr(p.status, topk_bits);
  }
#ifdef MLA_TRACE
  __syncthreads();
  if (tid == 0) g_mla_kernel_times[1] = globaltimer_ns();
#endif
}

// ---------------------------------------------------------------- K0b
// e4m3 cache: per query row r of request b, the scale of its e4m3 split,
// max |q| / 448 over the 576 values (1 for an all-zero row), and (with
// p.qterms) the split itself: hi = e4m3(q / scale), lo = e4m3(q / scale -
// hi), 576 codes each, the same arithmetic as the attention kernel's own
// split.  One warp per row.
__device__ __forceinline__ void e4m3_split_pair(float2 x, uint32_t& hi16, uint32_t& lo16) {
  const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
  const __nv_fp8x2_storage_t l = __nv_cvt_float2_to_fp8x2(make_float2(x.x - hf.x, x.y - hf.y), __NV_SATFINITE, __NV_E4M3);
  hi16 = h;
  lo16 = l;
}

__global__ void __launch_bounds__(256) mla_qscale_kernel(Params p) {
  // needs nothing from the schedule, so it may run beside it; block 0 ends
  // only after the schedule has (griddep_wait below), so the attention
  // kernel's wait for this grid covers both.  The other blocks leave as soon
  // as they are done: had each of them waited, the first waves would hold
  // their SMs until the schedule ended and the later ones would queue.
  griddep_launch_dependents();
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(p.B) * p.R) {
    if (blockIdx.x == 0) griddep_wait();
    return;
  }
  const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + row * kDL * 2);
  const uint4* qp = reinterpret_cast<const uint4*>(p.q_pe + row * kDR * 2);
  // the row's 72 chunks of 16 bytes: all of a lane's loads in flight at once
  uint4 v[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int c = lane + 32 * k;
    v[k] = c < 64 ? __ldg(qn + c) : (c < 72 ? __ldg(qp + (c - 64)) : make_uint4(0u, 0u, 0u, 0u));
  }
  float amax = 0.f;  // zero chunks leave the maximum of |q| unchanged
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const uint32_t ws[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[e]));
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float qs = amax > 0.f ? amax / 448.f : 1.f;  // every lane holds the row's max
  if (lane == 0) p.qscale[row] = qs;
  if (p.qterms) {  // chunk c (8 values) -> 8 hi codes at 8c, 8 lo codes at 576 + 8c
    const float inv = 1.f / qs;
    uint8_t* t = p.qterms + row * 1152;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int c = lane + 32 * k;
      if (c >= 72) continue;
      const uint32_t ws[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      uint32_t hi[2], lo[2];
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[2 * h2]));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[2 * h2 + 1]));
        uint32_t h0, l0, h1, l1;
        e4m3_split_pair(make_float2(f0.x * inv, f0.y * inv), h0, l0);
        e4m3_split_pair(make_float2(f1.x * inv, f1.y * inv), h1, l1);
        hi[h2] = (h0 & 0xFFFFu) | (h1 << 16);
        lo[h2] = (l0 & 0xFFFFu) | (l1 << 16);
      }
      *reinterpret_cast<uint2*>(t + 8 * c) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(t + 576 + 8 * c) = make_uint2(lo[0], lo[1]);
    }
  }
  if (blockIdx.x == 0) griddep_wait();
}

// One request's piece inside a cluster's slice.
struct Unit {
  int b, p0, p1, np, L, slot;  // slot < 0: the piece is the whole request
};

struct UnitIter {
  const int32_t* prefix;
  const int32_t* seq_lens;
  int B, s, e, b, bfirst, cid, max_pages, len_offset, len_fixed;
  __device__ void init(const Params& p, int c) {
    prefix = p.prefix;
    seq_lens = p.seq_lens;
    len_offset = p.len_offset;
    len_fixed = p.len_fixed;
    B = p.B;
    max_pages = p.max_pages;
    cid = c;
    s = p.cinfo[3 * c + 0];
    e = p.cinfo[3 * c + 1];
    bfirst = p.cinfo[3 * c + 2];
    b = bfirst;
  }
  __device__ bool next(Unit& u) {
    while (b < B && s < e) {
      const int pb0 = prefix[b];
      if (pb0 >= e) return false;
      const int pb1 = prefix[b + 1];
      const int p0 = (s > pb0 ? s : pb0) - pb0;
      const int p1 = (e < pb1 ? e : pb1) - pb0;
      const int bb = b++;
      if (p1 > p0) {
        u.b = bb;
        u.p0 = p0;
        u.p1 = p1;
        u.np = pb1 - pb0;
        u.L = clamp_len(req_len(seq_lens, bb, len_offset, len_fixed), max_pages);
        u.slot = (p0 > 0 || p1 < u.np) ? 2 * cid + (bb != bfirst ? 1 : 0) : -1;
        return true;
      }
    }
    return false;
  }
};

// Which wait gave up, recorded (first one only) in status[1..3] of the
// workspace: wait tag, page counter, (cluster << 16) | (rank << 8) | warp.
enum WaitTag : int {
  kWaitProdEmptyS = 1, kWaitProdEmptyO, kWaitQFull, kWaitKvFullS, kWaitSEmpty, kWaitSFull, kWaitPEmptyS,
  kWaitMlEmpty, kWaitKvFullO, kWaitPFullO, kWaitOEmpty, kWaitRescDone, kWaitPFullCorr, kWaitPvPrev,
  kWaitOFull, kWaitMlFull, kWaitSPrevUnit, kWaitPvReady, kWaitPvTaken, kWaitQEntry, kWaitPub
};

__device__ __forceinline__ void raise_timeout(const Params& p, Ctrl* ctrl, uint32_t partner_rank, int tag,
                                              uint32_t j) {
  if (atomicCAS(p.status + 1, 0, tag) == 0) {
    p.status[2] = static_cast<int32_t>(j);
    p.status[3] = static_cast<int32_t>((cluster_id_x() << 16) | (cluster_ctarank() << 8) | (threadIdx.x >> 5));
  }
  atomicOr(p.status, MLA_DEV_TIMEOUT);
  *reinterpret_cast<volatile int*>(&ctrl->abort) = 1;
  st_cluster_u32(mapa(smem_u32(&ctrl->abort), partner_rank), 1u);
}

__device__ __forceinline__ int32_t read_page_id(const Params& p, int b, int pg) {
  const int32_t pid = __ldg(p.page_table + static_cast<int64_t>(b) * p.pt_stride + pg);
  if (pid < 0 || pid >= p.num_pages) {
    atomicOr(p.status, MLA_DEV_BAD_PAGE_ID);
    return 0;
  }
  return pid;
}

// Ring entries of the bf16 S CTA holding a unit's query rows: 64 rows per
// entry, laid out like a page (8 boxes of q_nope, the 9th of q_pe).
__device__ __forceinline__ int q_entries(int rows_real) { return (rows_real + 63) / 64; }
// Ring entries of the S CTA holding a unit's query rows: bf16, 64 rows per
// entry; e4m3 terms (hi + lo, 1152 bytes a row like bf16), 32 rows per
// 36 KB entry (kQT); none when the e4m3 kernel splits the rows itself.
template <bool kF8, bool kQT>
__device__ __forceinline__ int q_entries_of(int rows_real) {
  return kF8 ? (kQT ? (rows_real + 31) / 32 : 0) : q_entries(rows_real);
}

// TMA producer shared by both roles: streams the slice's pages into a ring
// of kNSt slots (entry i: slot i % kNSt, phase (i / kNSt) & 1).  The bf16 S
// CTA streams, ahead of each unit's pages, the unit's query rows as well
// (q_entries entries), which the softmax warps move into TMEM: coalesced
// copies issued as soon as a slot frees, instead of per-row loads at the
// unit boundary.
template <bool kF8, bool kQT, bool kRoleS>
__device__ void run_producer(const Params& p, Ctrl* ctrl, uint8_t* ring, const CUtensorMap* tm_kv,
                             const CUtensorMap* tm_pe, const CUtensorMap* tm_qn, const CUtensorMap* tm_qp, int cid,
                             int g, uint32_t partner) {
  using C = Cfg<kF8>;
  constexpr int kNSt = kRoleS ? C::kNStS : C::kNStO;
  constexpr int kSlot = kRoleS ? C::kSlotS : C::kSlotO;
  constexpr uint32_t kCopyBytes = static_cast<uint32_t>((kRoleS ? C::kBoxesPartS : C::kBoxesPartO) * C::kBox);
  volatile int* abort = &ctrl->abort;
  const int rows_real = p.R - g * kRows < kRows ? p.R - g * kRows : kRows;
  const int qe = kRoleS ? q_entries_of<kF8, kQT>(rows_real) : 0;
  UnitIter it;
  it.init(p, cid);
  Unit u;
  uint32_t j = 0;  // pages
  uint32_t i = 0;  // ring entries
  bool ok = true;
  // waits for the slot of entry i; returns its full barrier and address
  auto acquire = [&](uint32_t& bar, uint8_t*& slot) -> bool {
    const int st = static_cast<int>(i % kNSt);
    if (!mbar_wait(smem_u32(&ctrl->kv_empty[st]), ((i / kNSt) & 1) ^ 1, abort, p.timeout_ns)) {
      raise_timeout(p, ctrl, partner, kRoleS ? kWaitProdEmptyS : kWaitProdEmptyO, j);
      return false;
    }
    bar = smem_u32(&ctrl->kv_full[st]);
    slot = ring + st * kSlot;
    return true;
  };
  // the next unit's query rows are pulled into L2 as well
  UnitIter nxt;
  nxt.init(p, cid);
  Unit un_next;
  bool have_next = kRoleS && nxt.next(un_next);
  auto prefetch_q = [&](const Unit& w) {
    const int64_t row0 = static_cast<int64_t>(w.b) * p.Q * p.H + g * kRows;
    prefetch_l2_bulk(p.q_nope + row0 * kDL * 2, static_cast<uint32_t>(rows_real) * kDL * 2);
    prefetch_l2_bulk(p.q_pe + row0 * kDR * 2, static_cast<uint32_t>(rows_real) * kDR * 2);
  };
  if (have_next) prefetch_q(un_next);
  while (ok && it.next(u)) {
    // the next unit's query rows are pulled into L2 when this unit has a
    // few pages left to copy (~10 pages before they are read): issued at the
    // unit's start, a long unit's page stream evicted them again
    if (kRoleS) have_next = have_next && nxt.next(un_next);
    const int pf_page = u.p1 - 4 > u.p0 ? u.p1 - 4 : u.p0;
    for (int e = 0; e < qe && ok; ++e) {
      uint32_t bar;
      uint8_t* slot;
      if (!acquire(bar, slot)) {
        ok = false;
        break;
      }
      const int row = static_cast<int>(static_cast<int64_t>(u.b) * p.Q * p.H + g * kRows + (kF8 ? 32 : 64) * e);
      mbar_expect_tx(bar, static_cast<uint32_t>(C::kSlotS));
      tma_load_3d(smem_u32(slot), tm_qn, 0, row, 0, bar);  // e4m3: the 9 boxes of 32 rows of terms
      if constexpr (!kF8) tma_load_2d(smem_u32(slot + C::kNBoxLat * C::kBox), tm_qp, 0, row, bar);
      ++i;
    }
    for (int pg = u.p0; pg < u.p1 && ok; ++pg, ++j) {
      if (kRoleS && have_next && pg == pf_page) prefetch_q(un_next);
      const int32_t pid = read_page_id(p, u.b, pg);
      const int y = pid * kPage;
      uint32_t bar;
      uint8_t* slot;
      if (!acquire(bar, slot)) {
        ok = false;
        break;
      }
      const bool pe = kRoleS && kF8;  // e4m3 S CTA: the k_pe box comes by its own map
      mbar_expect_tx(bar, kCopyBytes + (pe ? static_cast<uint32_t>(C::kPeBytes) : 0u));
      // one 3-D box: 128-byte columns x 64 token rows, box-major, 128-byte swizzled
      tma_load_3d(smem_u32(slot), tm_kv, 0, y, 0, bar);
      if (pe) tma_load_2d(smem_u32(slot + C::kNBoxLat * C::kBox), tm_pe, kDL, y, bar);
      ++i;
      MLA_TRACE_POINT(kRoleS ? 0 : 1, 0, j);
    }
  }
  // Drain: every copy issued into each slot must have landed before exit.
  for (uint32_t q = 0; q < static_cast<uint32_t>(kNSt) && q < i; ++q) {
    const uint32_t last = i - 1 - ((i - 1 - q) % kNSt);  // last entry in slot q
    const uint32_t ph = (last / kNSt) & 1;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(&ctrl->kv_full[q]), ph) && globaltimer_ns() - t0 < p.timeout_ns) {
    }
  }
}

// Writes one row's final (unsplit) or partial (split) result.
// Columns [256 * half, 256 * half + 256) of the row; half 0 also writes the lse.
template <bool kF8>
__device__ __forceinline__ void store_row(const Params& p, const Unit& u, int g, int r, int half,
                                          uint32_t taddr_row, float m_log2, float l) {
  const int rr = g * kRows + r;
  const bool real = rr < p.R;
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
  const float oscale = kF8 ? p.kv_scale * inv_l : inv_l;
  const float lse_v = l > 0.f ? (m_log2 - SoftmaxCfg<kF8>::kShift + __log2f(l)) * kLn2 : -INFINITY;
  if (u.slot >= 2 * p.C || u.b >= p.B) {  // cannot happen; checked so a bad schedule never writes out of range
    atomicOr(p.status, MLA_DEV_INTERNAL);
    return;
  }
  if (u.slot < 0 && p.out_f32) {  // unsplit, fp32 output: the values of a partial
    const int i = rr / p.H, h = rr % p.H;
    const int64_t orow = (static_cast<int64_t>(u.b) * p.Q + i) * p.H + h;
    float4* dst = reinterpret_cast<float4*>(p.out + orow * kDL * 4);
#pragma unroll 1
    for (int c = half * 256; c < half * 256 + 256; c += 32) {
      uint32_t v[2][16];
      tmem_ld16(taddr_row + c, v[0]);
      tmem_ld16(taddr_row + c + 16, v[1]);
      tmem_wait_ld_tie(v[0]);
      tmem_wait_ld_tie(v[1]);
      if (real) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[q][8 * k + e]) * oscale);
            stg_v8(dst + (c + 16 * q) / 4 + 2 * k, w);  // 8 floats = 32 bytes
          }
      }
    }
    if (real && half == 0) p.lse[orow] = lse_v;
  } else if (u.slot < 0) {
    const int i = rr / p.H, h = rr % p.H;
    const int64_t orow = (static_cast<int64_t>(u.b) * p.Q + i) * p.H + h;
    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * kDL * 2);
#pragma unroll 1
    for (int c = half * 256; c < half * 256 + 256; c += 32) {  // two TMEM loads in flight per wait
      uint32_t v[2][16];
      tmem_ld16(taddr_row + c, v[0]);
      tmem_ld16(taddr_row + c + 16, v[1]);
      tmem_wait_ld_tie(v[0]);
      tmem_wait_ld_tie(v[1]);
      if (real) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[q][2 * k]) * oscale,
                                                      __uint_as_float(v[q][2 * k + 1]) * oscale);
            w[k] = *reinterpret_cast<uint32_t*>(&b2);
          }
          stg_v8(dst + (c + 16 * q) / 8, w);  // 16 bf16 = 32 bytes
        }
      }
    }
    if (real && half == 0) p.lse[orow] = lse_v;
  } else {
    const int64_t prow = (static_cast<int64_t>(u.slot) * p.G + g) * kRows + r;
    float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kDL);
#pragma unroll 1
    for (int c = half * 256; c < half * 256 + 256; c += 32) {
      uint32_t v[2][16];
      tmem_ld16(taddr_row + c, v[0]);
      tmem_ld16(taddr_row + c + 16, v[1]);
      tmem_wait_ld_tie(v[0]);
      tmem_wait_ld_tie(v[1]);
      if (real) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[q][8 * k + e]) * oscale);
            stg_v8(dst + (c + 16 * q) / 4 + 2 * k, w);  // 8 floats = 32 bytes
          }
      }
    }
    if (real && half == 0) p.lse_part[prow] = lse_v;
  }
}

// Loads the 16-byte chunks [c0, c0 + kN) of query row r of row block g for
// request b (chunk c = 8 values: c < 64 from q_nope, else q_pe) into TMEM
// lane r, packed along K: 2 bf16 or 4 e4m3 per column.  e4m3: both terms
// of the split with the row's scale qs_in, which is returned.
template <bool kF8, int kN = 72>
__device__ __forceinline__ float load_q_row(const Params& p, int b, int g, int r, uint32_t taddr_row, int c0 = 0,
                                            float qs_in = 1.f) {
  const int rr = g * kRows + r;
  const bool real = rr < p.R;
  const uint4* qn = nullptr;
  const uint4* qp = nullptr;
  if (real) {
    const int i = rr / p.H, h = rr % p.H;
    const int64_t row = (static_cast<int64_t>(b) * p.Q + i) * p.H + h;
    qn = reinterpret_cast<const uint4*>(p.q_nope + row * kDL * 2);
    qp = reinterpret_cast<const uint4*>(p.q_pe + row * kDR * 2);
  }
  // chunks c, c + 1 (c even; chunk = 8 bf16 values) as one 32-byte load
  auto pair = [&](int c, uint32_t (&w)[8]) {
    if (!real) {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = 0u;
    } else {
      ldg_v8(c < 64 ? static_cast<const void*>(qn + c) : static_cast<const void*>(qp + (c - 64)), w);
    }
  };
  if constexpr (!kF8) {
    static_assert(kN % 12 == 0, "rounds of 12 chunks");
#pragma unroll
    for (int c = 0; c < kN; c += 12) {
      uint32_t v[6][8];
#pragma unroll
      for (int k = 0; k < 6; ++k) pair(c0 + c + 2 * k, v[k]);
#pragma unroll
      for (int s4 = 0; s4 < 3; ++s4) {
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          w[e] = v[2 * s4][e];
          w[8 + e] = v[2 * s4 + 1][e];
        }
        tmem_st16(taddr_row + (c0 + c + 4 * s4) * 4, w);
      }
    }
    tmem_wait_st();
    return 1.f;
  } else {
    // e4m3: chunks [c0, c0 + kN) (kN a multiple of 8) as hi + lo terms with
    // the row's scale qs_in (value = code * qs)
    const float qs = qs_in;
    const float inv = 1.f / qs;
    // two e4m3 codes for a pair of scaled values: hi = e4m3(x), lo = e4m3(x - hi)
    auto split2 = [](float2 x, uint32_t& hi16, uint32_t& lo16) {
      const __nv_fp8x2_storage_t h = __nv_cvt_float2_to_fp8x2(x, __NV_SATFINITE, __NV_E4M3);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
      const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_fp8x2_storage_t l =
          __nv_cvt_float2_to_fp8x2(make_float2(x.x - hf.x, x.y - hf.y), __NV_SATFINITE, __NV_E4M3);
      hi16 = h;
      lo16 = l;
    };
    static_assert(kN % 8 == 0, "rounds of 8 chunks");
    // rounds of 64 values (16 columns of each term); the loads of round n + 1
    // are issued before round n is converted, so that one global-load
    // latency is exposed per row instead of one per round
    uint32_t nxt[4][8];
#pragma unroll
    for (int k = 0; k < 4; ++k) pair(c0 + 2 * k, nxt[k]);
#pragma unroll
    for (int c = c0; c < c0 + kN; c += 8) {
      uint32_t v8[4][8];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[k][e] = nxt[k][e];
      if (c + 8 < c0 + kN) {
#pragma unroll
        for (int k = 0; k < 4; ++k) pair(c + 8 + 2 * k, nxt[k]);
      }
      uint32_t whi[16], wlo[16];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t ws[4] = {v8[k >> 1][4 * (k & 1)], v8[k >> 1][4 * (k & 1) + 1], v8[k >> 1][4 * (k & 1) + 2],
                                v8[k >> 1][4 * (k & 1) + 3]};
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[2 * h2]));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[2 * h2 + 1]));
          uint32_t h0, l0, h1, l1;
          split2(make_float2(f0.x * inv, f0.y * inv), h0, l0);
          split2(make_float2(f1.x * inv, f1.y * inv), h1, l1);
          whi[2 * k + h2] = (h0 & 0xFFFFu) | (h1 << 16);
          wlo[2 * k + h2] = (l0 & 0xFFFFu) | (l1 << 16);
        }
      }
      tmem_st16(taddr_row + c * 2, whi);
      tmem_st16(taddr_row + Cfg<kF8>::kQLoCol + c * 2, wlo);
    }
    tmem_wait_st();
    return qs;
  }
}

// A query row from a ring entry into TMEM lane r: 16-byte chunks [c0, c0 +
// 36) (chunk c = box c / 8, piece c % 8 of the 128-byte-swizzled row rq;
// boxes of kBoxBytes).  bf16: 8 boxes of q_nope, then q_pe, 2 values a
// column; e4m3: the row's hi term then its lo term, 4 codes a column, so the
// lo term starts at column 144.  src = the row's first box row, or null for
// a padding row (zeros).
template <int kBoxBytes>
__device__ __forceinline__ void load_q_row_smem(const uint8_t* src, int rq, uint32_t taddr_row, int c0) {
#pragma unroll
  for (int c = 0; c < 36; c += 12) {
    uint4 v[12];
#pragma unroll
    for (int k = 0; k < 12; ++k) {
      const int cc = c0 + c + k;
      v[k] = src ? *reinterpret_cast<const uint4*>(src + (cc >> 3) * kBoxBytes + (((cc & 7) ^ (rq & 7)) << 4))
                 : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int s4 = 0; s4 < 3; ++s4) {
      const uint32_t w[16] = {v[4 * s4].x,     v[4 * s4].y,     v[4 * s4].z,     v[4 * s4].w,
                              v[4 * s4 + 1].x, v[4 * s4 + 1].y, v[4 * s4 + 1].z, v[4 * s4 + 1].w,
                              v[4 * s4 + 2].x, v[4 * s4 + 2].y, v[4 * s4 + 2].z, v[4 * s4 + 2].w,
                              v[4 * s4 + 3].x, v[4 * s4 + 3].y, v[4 * s4 + 3].z, v[4 * s4 + 3].w};
      tmem_st16(taddr_row + (c0 + c + 4 * s4) * 4, w);
    }
  }
  tmem_wait_st();
}

// ---------------------------------------------------------------- K1
// kQT (e4m3 only): the query terms come from the scale pre-pass through the
// ring (p.qterms), else the softmax warps split the bf16 rows themselves;
// separate instantiations, so that neither path's registers burden the other.
template <bool kF8, bool kQT>
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_s,
                      const __grid_constant__ CUtensorMap tm_o, const __grid_constant__ CUtensorMap tm_pe,
                      const __grid_constant__ CUtensorMap tm_qn, const __grid_constant__ CUtensorMap tm_qp) {
  using C = Cfg<kF8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* data = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(data + C::kData);
  // one S/O pair per cluster; cluster k computes row block g = k mod G of
  // slice k / G (the pairs of a slice share nothing but the pages they read)
  const uint32_t rank = cluster_ctarank();
  const bool role_s = rank == 0;
  const uint32_t partner = rank ^ 1u;
  const int clus = static_cast<int>(cluster_id_x());
  const int g = clus % p.G;
  const int cid = clus / p.G;  // the slice
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#ifdef MLA_TRACE
  if (threadIdx.x == 0) atomicMin(&g_mla_kernel_times[4], globaltimer_ns());
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < 6; ++i) {
      mbar_init(smem_u32(&ctrl->kv_full[i]), 1);
      mbar_init(smem_u32(&ctrl->kv_empty[i]), 1);
    }
    for (int i = 0; i < kNS; ++i) {
      mbar_init(smem_u32(&ctrl->s_full[i]), 1);
      mbar_init(smem_u32(&ctrl->s_empty[i]), kRowWarps / 2);  // the group that read the page
    }
    mbar_init(smem_u32(&ctrl->q_full), kRowWarps);  // both groups load the queries
    for (int i = 0; i < kMaxPSlots; ++i) {
      mbar_init(smem_u32(&ctrl->p_full[i]), 1);  // one arm (expect_tx) by the O MMA warp + P bytes
      mbar_init(smem_u32(&ctrl->p_empty[i]), 1);
    }
    mbar_init(smem_u32(&ctrl->resc_req), 1);
    mbar_init(smem_u32(&ctrl->resc_done), kRowWarps);
    mbar_init(smem_u32(&ctrl->o_full), 1);
    mbar_init(smem_u32(&ctrl->o_empty), kRowWarps);
    mbar_init(smem_u32(&ctrl->ml_full), kRowWarps);
    mbar_init(smem_u32(&ctrl->ml_empty), kRowWarps);
    mbar_init(smem_u32(&ctrl->pv_ready), 1);
    mbar_init(smem_u32(&ctrl->pv_taken), 1);
    mbar_init(smem_u32(&ctrl->drain), 1);
    ctrl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(role_s ? &tm_s : &tm_o);
    if constexpr (kF8) tma_prefetch_desc(&tm_pe);
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(&ctrl->tmem_base), 512);
    tmem_relinquish();
  }
  if (role_s && threadIdx.x >= 128)  // page references: no page yet
    for (int i = threadIdx.x - 128; i < 4 * kRows; i += blockDim.x - 128)
      reinterpret_cast<uint64_t*>(data + C::kPubOff)[i] = 0ull;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // partner barriers initialised before any remote arrive
  // everything above overlaps the end of the kernel before this one; the
  // schedule (and the e4m3 query scales) are read only after it completed
  griddep_wait();
  griddep_launch_dependents();  // the combine may launch as clusters finish
  const uint32_t tmem = ctrl->tmem_base;
  volatile int* abort = &ctrl->abort;
#ifdef MLA_TRACE
  if (threadIdx.x == 0 && rank == 0 && clus < 1024) g_mla_cluster_times[clus][0] = globaltimer_ns();
  if (threadIdx.x == 0) atomicMin(&g_mla_kernel_times[5], globaltimer_ns());
#endif

  if (role_s) {
    // =========================== S CTA ===========================
    uint8_t* ring = data;
    if (warp == 0) {
      if (lane == 0) run_producer<kF8, kQT, true>(p, ctrl, ring, &tm_s, &tm_pe, &tm_qn, &tm_qp, cid, g, partner);
    } else if (warp == 1) {
      // QK issuer: the whole warp runs the loop and one elected lane issues
      // (a converged warp keeps the tensor pipe full with N = 64 MMAs), so
      // each page's 36 MMAs run back to back and its ring slot frees early
      UnitIter it;
      it.init(p, cid);
      Unit u;
      uint32_t j = 0, un = 0;
      bool ok = true;
      int why = 0;
      const int qe = q_entries_of<kF8, kQT>(p.R - g * kRows < kRows ? p.R - g * kRows : kRows);
      while (ok && it.next(u)) {
        if (!mbar_wait_warp(smem_u32(&ctrl->q_full), un & 1, abort, p.timeout_ns)) {
          ok = false;
          why = kWaitQFull;
          break;
        }
        // the unit's query entries were moved into TMEM: their slots go back
        // to the producer (entries j + qe * un ..)
        for (int e = 0; e < qe; ++e)
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->kv_empty[(j + qe * un + e) % C::kNStS]));
        ++un;
        for (int pg = u.p0; pg < u.p1; ++pg, ++j) {
          const uint32_t ri = j + qe * un;  // ring entry of this page
          const int st = ri % C::kNStS;
          const int sb = j % kNS;
          const uint32_t kph = (ri / C::kNStS) & 1;
          if (lane == 0) MLA_TRACE_POINT(0, 9, j);
          {  // S buffer free and page landed, polled together
            const uint32_t bars[4] = {smem_u32(&ctrl->s_empty[sb]), smem_u32(&ctrl->kv_full[st]), 0u, 0u};
            const uint32_t pars[4] = {((j / kNS) & 1) ^ 1, kph, 0u, 0u};
            if (!mbar_wait4_warp(bars, pars, abort, p.timeout_ns)) {
              ok = false;
              why = kWaitKvFullS;
              break;
            }
          }
          if (lane == 0) MLA_TRACE_POINT(0, 1, j);
          tc_fence_after();
          // descriptors of box 0 / the k_pe box at K step 0; a K step adds
          // 32 bytes (2 in the >>4 address field), a box adds 8 KB (512)
          const uint32_t slot_addr = smem_u32(ring + st * C::kSlotS);
          const uint64_t dlat = smem_desc(slot_addr, 16, 1024, kSwizzle128B);
          const uint32_t dcol = tmem + kSCol0 + sb * 64;
          if constexpr (!kF8) {
            // 9 boxes (8 of c_kv, 1 of k_pe) x 4 K steps
#pragma unroll
            for (int d = 0; d < 9; ++d)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ts_e<false>(dcol, tmem + d * 32 + k * 8, dlat + static_cast<uint64_t>(d * 512 + k * 2),
                                C::kIdescQK, (d | k) ? 1u : 0u);
          } else {
            const uint64_t dpe = smem_desc(slot_addr + C::kNBoxLat * C::kBox, 16, C::kPeSbo, C::kPeSwz);
#pragma unroll
            for (int term = 0; term < C::kQSplit; ++term) {
              const uint32_t qcol = tmem + (term ? C::kQLoCol : 0u);
#pragma unroll
              for (int d = 0; d < C::kNBoxLat; ++d)
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  mma_ts_e<true>(dcol, qcol + d * 32 + k * 8, dlat + static_cast<uint64_t>(d * 512 + k * 2),
                                 C::kIdescQK, (term | d | k) ? 1u : 0u);
#pragma unroll
              for (int k = 0; k < C::kKStepsPe; ++k)
                mma_ts_e<true>(dcol, qcol + C::kNBoxLat * 32 + k * 8, dpe + static_cast<uint64_t>(k * 2),
                               C::kIdescQK, 1u);
            }
          }
          mma_commit_e(smem_u32(&ctrl->kv_empty[st]));
          mma_commit_e(smem_u32(&ctrl->s_full[sb]));
          if (lane == 0) MLA_TRACE_POINT(0, 2, j);
        }
      }
      if (!ok && lane == 0) raise_timeout(p, ctrl, partner, why, j);
      mma_commit_e(smem_u32(&ctrl->drain));
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctrl->drain), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
        }
      }
      __syncwarp();
    } else if (warp >= 4) {
      // ---- softmax: group gg (warps 4-7: 0, warps 8-11: 1) takes the pages
      // j with j % 2 == gg; its thread r owns query row r.  P of a page is
      // computed against a reference (a running max of the row) that is
      // sent with it; the O CTA brings every page to one frame.  A page's
      // reference is the previous page's, raised to the page max when that
      // exceeds it by more than a threshold; each page publishes its own.
      // So references are a function of the data alone (results do not
      // depend on timing) and never fall within a unit; a page waits only
      // for the previous page's row max, not for its P.
      // Each group keeps its partial sum in the frame of its latest reference.
      const int r = (warp & 3) * 32 + lane;
      const int gg = (warp - 4) >> 2;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t p_remote = mapa(smem_u32(data + C::kPOff), partner);
      const uint32_t ref_remote = mapa(smem_u32(data + C::kRefOff), partner);
      const uint32_t flag_remote = mapa(smem_u32(data + C::kFlagOff), partner);
      const uint32_t mlfull_remote = mapa(smem_u32(&ctrl->ml_full), partner);
      volatile uint64_t* pub = reinterpret_cast<volatile uint64_t*>(data + C::kPubOff);
      const int rr = g * kRows + r;
      const bool real = rr < p.R;  // rows past H * q_len are padding: nothing of theirs is sent
      const PSlots ps(kF8, p.R - g * kRows < kRows ? p.R - g * kRows : kRows);
      const int qi = real ? rr / p.H : p.Q - 1;
      const int qe = q_entries_of<kF8, kQT>(p.R - g * kRows < kRows ? p.R - g * kRows : kRows);
      UnitIter it;
      it.init(p, cid);
      Unit u;
      uint32_t j = 0, un = 0;
      bool ok = true;
      int why = 0;
      while (ok && it.next(u)) {
        // both groups load part of every query row (e4m3: with the row's scale
        // from the pre-pass)
        const float qs = (kF8 && real) ? p.qscale[static_cast<int64_t>(u.b) * p.R + rr] : 1.f;
        if (r == 0 && gg == 0) MLA_TRACE_POINT(0, 11, un);
        {
          // the queries of this unit replace the previous unit's in TMEM once
          // every QK of that unit is done: the S of its last page has landed
          // (one issuer: its commit covers all its earlier MMAs)
          if (j > 0 && !mbar_wait_warp<false, true>(smem_u32(&ctrl->s_full[(j - 1) % kNS]), ((j - 1) / kNS) & 1,
                                                    abort, p.timeout_ns)) {
            ok = false;
            why = kWaitSPrevUnit;
            break;
          }
          if (r == 0 && gg == 0) MLA_TRACE_POINT(0, 12, un);
          if constexpr (kF8 && !kQT) {
            if (gg == 0) load_q_row<true, 32>(p, u.b, g, r, tmem + lane_base, 0, qs);
            else load_q_row<true, 40>(p, u.b, g, r, tmem + lane_base, 32, qs);
          } else {
            // the producer copied this unit's query rows (e4m3: their terms)
            // into ring entries j + qe * un ..; half gg moves chunks
            // [36 gg, 36 gg + 36) of row r (e4m3: the hi, then the lo term)
            const uint32_t iq = j + qe * un;
            bool got = true;
            for (int e = 0; e < qe && got; ++e)
              got = mbar_wait_warp<false, true>(smem_u32(&ctrl->kv_full[(iq + e) % C::kNStS]),
                                                ((iq + e) / C::kNStS) & 1, abort, p.timeout_ns);
            if (!got) {
              ok = false;
              why = kWaitQEntry;
              break;
            }
            constexpr int kEntryRows = kF8 ? 32 : 64;
            const int e = r / kEntryRows, rq = r % kEntryRows;
            const uint8_t* src = (real && e < qe) ? ring + ((iq + e) % C::kNStS) * C::kSlotS + rq * 128 : nullptr;
            load_q_row_smem<kEntryRows * 128>(src, rq, tmem + lane_base, 36 * gg);
          }
          tc_fence_before();
          __syncwarp();
          // release the queries to the QK issuer
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->q_full));
          if (r == 0 && gg == 0) MLA_TRACE_POINT(0, 13, un);
        }
        const float c2 = p.scale * kLog2e * (kF8 ? qs * p.kv_scale : 1.f);  // log2-domain score scale
        const int nvis = u.L - p.Q + qi + 1;
        float m_run = kMinusBig, l = 0.f;  // this group's frame and partial sum
        for (int pg = u.p0; pg < u.p1; ++pg, ++j) {
          if ((j & 1u) != static_cast<uint32_t>(gg)) continue;
          const int sb = j % kNS;
          if (!mbar_wait_warp<false, true>(smem_u32(&ctrl->s_full[sb]), (j / kNS) & 1, abort, p.timeout_ns)) {
            ok = false;
            why = kWaitSFull;
            break;
          }
          if (r == 0) MLA_TRACE_POINT(0, 3, j);
          tc_fence_after();
          // S of the page, each load with the maximum of its 16 columns
          // (sm_103a's TMEM load with max-reduction)
          uint32_t v[4][16];
          float red[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) tmem_ld16_max(tmem + lane_base + kSCol0 + sb * 64 + q4 * 16, v[q4], red[q4]);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) tmem_wait_ld_tie(v[q4], red[q4]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->s_empty[sb]));
          if (r == 0) MLA_TRACE_POINT(0, 7, j);
          const int t0 = pg * kPage;
          // every key of the page visible to the row: no per-key masking
          const bool full = t0 + kPage <= nvis;
#define MLA_S(t) __uint_as_float(v[(t) >> 4][(t) & 15])
          // max of the raw scores (c2 > 0, so scaling commutes with max): on
          // a full page the loads' reduced values; otherwise masked here, so
          // that unused slots (even NaN) never count
          float m4[4] = {red[0], red[1], red[2], red[3]};
          if (!full) {
            m4[0] = m4[1] = m4[2] = m4[3] = -INFINITY;
#pragma unroll
            for (int t = 0; t < 64; ++t)
              if (t0 + t < nvis) m4[t & 3] = fmaxf(m4[t & 3], MLA_S(t));
          }
          const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2;
          // reference: the previous page's of the unit (entry (j - 1) % 4,
          // tagged j), raised to the page max when that exceeds it by more
          // than the threshold (P then stays <= 2^thr); published in entry
          // j % 4 with tag j + 1.  The entry is rewritten by page j + 3 only,
          // whose reference needs this page's, so no entry is overwritten
          // before it was read.
          float m_ref = m_run;
          float m_prev = kMinusBig;  // the previous page's reference: O's frame before this page
          if (pg != u.p0) {
            volatile uint64_t* pe = pub + ((j - 1u) & 3u) * kRows + r;
            uint64_t pv = *pe;
            if (static_cast<uint32_t>(pv >> 32) != j) {
              const uint64_t t_start = globaltimer_ns();
              while (static_cast<uint32_t>((pv = *pe) >> 32) != j) {
                if (*abort || globaltimer_ns() - t_start > p.timeout_ns) break;
              }
            }
            if (__any_sync(0xffffffffu, static_cast<uint32_t>(pv >> 32) != j)) {
              ok = false;
              why = kWaitPub;
              break;
            }
            m_prev = __uint_as_float(static_cast<uint32_t>(pv));
            m_ref = fmaxf(m_ref, m_prev);
          }
          if (mx > m_ref + SoftmaxCfg<kF8>::kThreshold) m_ref = mx;
          pub[(j & 3u) * kRows + r] = (static_cast<uint64_t>(j + 1u) << 32) | __float_as_uint(m_ref);
          // O holds the earlier pages in the frame m_prev: when the reference
          // rose, O is scaled by o_scale before this page's PV (a unit's
          // first page sets the frame: its PV overwrites O)
          const bool rose = pg != u.p0 && m_ref > m_prev;
          const float o_scale = rose ? ex2_approx(m_prev - m_ref) : 1.f;
          const uint32_t rose_mask = __ballot_sync(0xffffffffu, rose && real);
          if (r == 0) MLA_TRACE_POINT(0, 8, j);
          l *= ex2_approx(m_run - m_ref);  // m_run <= m_ref: the partial sum moves to the new frame
          m_run = m_ref;
          // P (swizzled for the MMA) goes 16 bytes at a time into the O CTA's
          // shared memory, completing bytes on its p_full barrier, once P
          // slot ps_slot is free (the O CTA finished PV of page j - ps.n);
          // then the row's reference.  bf16: P is computed into registers
          // before the slot is waited for, which takes P's arithmetic off the
          // slot's round trip (blocks of more than 64 rows have two slots:
          // measured 5-11 % faster).  e4m3 (three slots, never waited for
          // long): each chunk is sent as soon as it is computed, so the
          // stores overlap the arithmetic (measured 1 % faster than the other
          // order).
          const int ps_slot = static_cast<int>(j % static_cast<uint32_t>(ps.n));
          const uint32_t ps_phase = (j / static_cast<uint32_t>(ps.n)) & 1;
          const float nm = SoftmaxCfg<kF8>::kShift - m_ref;  // P = 2^(s * c2 - m_ref + shift)
          auto prob = [&](int t) {
            const float e = ex2_approx(fmaf(MLA_S(t), c2, nm));
            return (full || t0 + t < nvis) ? e : 0.f;
          };
          const uint32_t bar = mapa(smem_u32(&ctrl->p_full[ps_slot]), partner);
          const uint32_t prow = p_remote + ps_slot * ps.stride + (r >> 3) * C::kPSbo + (r & 7) * 16;
          float s4[4] = {0.f, 0.f, 0.f, 0.f};
          if constexpr (!kF8) {
            uint4 pw[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) {  // keys 8c .. 8c + 7
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float a = prob(8 * c + 2 * k), b = prob(8 * c + 2 * k + 1);
                s4[k] += a + b;  // bf16 rounding of P changes l by < 2^-9 relative
                __nv_bfloat162 b2 = __floats2bfloat162_rn(a, b);
                w[k] = *reinterpret_cast<uint32_t*>(&b2);
              }
              pw[c] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (!mbar_wait_warp<true, true>(smem_u32(&ctrl->p_empty[ps_slot]), ps_phase ^ 1, abort, p.timeout_ns)) {
              ok = false;
              why = kWaitPEmptyS;
              break;
            }
            if (r == 0) MLA_TRACE_POINT(0, 4, j);
            if (real) {
#pragma unroll
              for (int c = 0; c < 8; ++c) st_async_v4(prow + c * C::kPLbo, pw[c], bar);
            }
          } else {
            if (!mbar_wait_warp<true, true>(smem_u32(&ctrl->p_empty[ps_slot]), ps_phase ^ 1, abort, p.timeout_ns)) {
              ok = false;
              why = kWaitPEmptyS;
              break;
            }
            if (r == 0) MLA_TRACE_POINT(0, 4, j);
#pragma unroll
            for (int c = 0; c < 4; ++c) {  // keys 16c .. 16c + 15
              uint32_t wh[4], wl[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int t = 16 * c + 4 * k;
                const float2 pa = make_float2(prob(t), prob(t + 1));
                const float2 pb = make_float2(prob(t + 2), prob(t + 3));
                // in f16 (e4m3 values convert to it exactly, and the residual
                // of an f16 value by its e4m3 rounding is exact in f16)
                const __half2 fa = __float22half2_rn(pa);
                const __half2 fb = __float22half2_rn(pb);
                const __nv_fp8x2_storage_t ha =
                    __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&fa), __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hb =
                    __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&fb), __NV_SATFINITE, __NV_E4M3);
                const __half2_raw xa = __nv_cvt_fp8x2_to_halfraw2(ha, __NV_E4M3);
                const __half2_raw xb = __nv_cvt_fp8x2_to_halfraw2(hb, __NV_E4M3);
                const __half2 ra = __hsub2(fa, *reinterpret_cast<const __half2*>(&xa));
                const __half2 rb = __hsub2(fb, *reinterpret_cast<const __half2*>(&xb));
                const __nv_fp8x2_storage_t la =
                    __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&ra), __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t lb =
                    __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&rb), __NV_SATFINITE, __NV_E4M3);
                // hi + lo equals p to about 2^-8 relative
                s4[k] += (pa.x + pa.y) + (pb.x + pb.y);
                wh[k] = static_cast<uint32_t>(ha) | (static_cast<uint32_t>(hb) << 16);
                wl[k] = static_cast<uint32_t>(la) | (static_cast<uint32_t>(lb) << 16);
              }
              if (real) {
                st_async_v4(prow + c * C::kPLbo, make_uint4(wh[0], wh[1], wh[2], wh[3]), bar);
                if constexpr (C::kPTerms > 1)
                  st_async_v4(prow + C::kPTermBytes + c * C::kPLbo, make_uint4(wl[0], wl[1], wl[2], wl[3]), bar);
              }
            }
          }
#undef MLA_S
          if (real) st_async_b32(ref_remote + (ps_slot * ps.arows + r) * 4, __float_as_uint(o_scale), bar);
          if (lane == 0) st_async_b32(flag_remote + (ps_slot * 4 + (warp & 3)) * 4, rose_mask, bar);
          l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
          if (r == 0) MLA_TRACE_POINT(0, 5, j);
        }
        if (!ok) break;
        // hand this group's (frame, partial sum) of the row to the O CTA
        if (!mbar_wait_warp<true, true>(smem_u32(&ctrl->ml_empty), (un & 1) ^ 1, abort, p.timeout_ns)) {
          ok = false;
          why = kWaitMlEmpty;
          break;
        }
        float* ml_buf = reinterpret_cast<float*>(data + C::kMlOff);
        ml_buf[4 * r + 2 * gg] = m_run;
        ml_buf[4 * r + 2 * gg + 1] = l;
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mlfull_remote);
        ++un;
      }
      if (!ok && lane == 0) raise_timeout(p, ctrl, partner, why, j);
    }
  } else {
    // =========================== O CTA ===========================
    uint8_t* ring = data + C::kRingOffO;
    uint8_t* pbuf = data + C::kPOff;
    const int rows_real = p.R - g * kRows < kRows ? p.R - g * kRows : kRows;
    const PSlots ps(kF8, rows_real);
    if (warp == 0) {
      if (lane == 0) run_producer<kF8, kQT, false>(p, ctrl, ring, &tm_o, &tm_pe, &tm_qn, &tm_qp, cid, g, partner);
    } else if (warp == 1) {
      // ---- PV warp: for page j it waits until the page is ready for PV
      // (c_kv landed, P arrived, O free on a unit's first page: the
      // independent conditions polled together), has O rescaled first when
      // a row's reference rose, zeroes the tail rows of a request's last
      // page, and issues PV(j); the whole warp runs the loop and one elected
      // lane issues.  (A separate waiter warp that prepared page j while
      // this one issued PV(j - 1) added a second poll between P's arrival
      // and its PV.)
      UnitIter it;
      it.init(p, cid);
      Unit u;
      uint32_t j = 0, un = 0;
      bool ok = true;
      int why = 0;
      const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << partner));
      // the S CTA sends the P rows (and O scale factors) of real query rows
      // only, and every softmax warp's flag word
      const uint32_t ptx = static_cast<uint32_t>(rows_real) * C::kPTxRow + C::kPTxFlags;
      const volatile uint32_t* flag_buf = reinterpret_cast<const volatile uint32_t*>(data + C::kFlagOff);
      uint32_t nreq = 0;  // rescale requests handed to the correction warps
      if (lane == 0) {  // arm the P barriers of the first pages (bytes may land before or after)
        for (int i = 0; i < ps.n; ++i) mbar_expect_tx(smem_u32(&ctrl->p_full[i]), ptx);
      }
      while (ok && it.next(u)) {
        for (int pg = u.p0; pg < u.p1; ++pg, ++j) {
          const int st = j % C::kNStO;
          const uint32_t kph = (j / C::kNStO) & 1;
          const int pb = static_cast<int>(j % static_cast<uint32_t>(ps.n));
          const uint32_t pph = (j / static_cast<uint32_t>(ps.n)) & 1;
          uint8_t* slot = ring + st * C::kSlotO;
          const bool first = pg == u.p0;
          if (lane == 0) MLA_TRACE_POINT(1, 8, j);
          {  // O free (a unit's first page), c_kv landed, P arrived
            const uint32_t bars[4] = {first ? smem_u32(&ctrl->o_empty) : 0u, smem_u32(&ctrl->kv_full[st]),
                                      smem_u32(&ctrl->p_full[pb]), 0u};
            const uint32_t pars[4] = {(un & 1) ^ 1, kph, pph, 0u};
            if (!mbar_wait4_warp(bars, pars, abort, p.timeout_ns)) {
              ok = false;
              why = kWaitPFullO;
              break;
            }
          }
          if (lane == 0) MLA_TRACE_POINT(1, 1, j);
          // a page on which some row's reference rose needs O rescaled first
          // (after PV(j - 1), the last one issued): the correction warps do it
          // and acknowledge
          const uint32_t fw = lane < 4 ? flag_buf[pb * 4 + lane] : 0u;
          if (__any_sync(0xffffffffu, fw != 0u)) {
            if (lane == 0) {
              ctrl->resc_page = j;
              mbar_arrive(smem_u32(&ctrl->resc_req));  // release: resc_page is seen with the phase
            }
            if (!mbar_wait_warp(smem_u32(&ctrl->resc_done), nreq & 1, abort, p.timeout_ns)) {
              ok = false;
              why = kWaitRescDone;
              break;
            }
            ++nreq;
          }
          // phase for page j done: arm this P slot for page j + ps.n.  Its
          // bytes cannot come earlier: the S CTA sends them only after PV(j)
          // ended.
          if (lane == 0) mbar_expect_tx(smem_u32(&ctrl->p_full[pb]), ptx);
          const int valid = u.L - pg * kPage;
          if (valid < kPage) {
            // token rows past the sequence end may hold anything (even NaN):
            // zero them so that P = 0 there cannot turn into 0 * NaN
            // lane: 16-byte chunk lane % 8 of rows v0 + lane / 8, + 4, ... in
            // every box (no division on the path to PV)
            const int v0 = valid > 0 ? valid : 0;
            const int chunk = lane & 7;
            for (int rowi = v0 + (lane >> 3); rowi < kPage; rowi += 4)
#pragma unroll
              for (int box = 0; box < C::kBoxesPartO; ++box)
                *reinterpret_cast<uint4*>(slot + box * C::kBox + rowi * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
            __syncwarp();
          }
          if (lane == 0) MLA_TRACE_POINT(1, 10, j);
          fence_proxy_async_cta();
          tc_fence_after();
          {  // the whole warp issues; one elected lane executes
            const uint64_t dv = smem_desc(smem_u32(ring + st * C::kSlotO), C::kBox, 1024, kSwizzle128B);
            // O[:, 256h .. 256h + 255] += P V[:, 256h ..], for each term of P
#pragma unroll
            for (int tm = 0; tm < C::kPTerms; ++tm) {
              const uint64_t dp =
                  smem_desc(smem_u32(pbuf + pb * ps.stride + tm * C::kPTermBytes), C::kPLbo, C::kPSbo, C::kPSwz);
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int k = 0; k < C::kPvKSteps; ++k)
                  mma_ss_e<kF8>(tmem + h * 256, dp + static_cast<uint64_t>(k * (2 * C::kPLbo >> 4)),
                                dv + static_cast<uint64_t>((h * C::kVBoxesHalf * C::kBox + k * C::kVKStepBytes) >> 4),
                                C::kIdescPV, (first && tm == 0 && k == 0) ? 0u : 1u);
            }
            mma_commit_e(smem_u32(&ctrl->kv_empty[st]));
            mma_commit_multicast_e(smem_u32(&ctrl->p_empty[pb]), mask);
            if (pg == u.p1 - 1) mma_commit_e(smem_u32(&ctrl->o_full));
            if (lane == 0) MLA_TRACE_POINT(1, 3, j);
          }
        }
        ++un;
      }
      if (!ok && lane == 0) raise_timeout(p, ctrl, partner, why, j);
      mma_commit_e(smem_u32(&ctrl->drain));
      if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&ctrl->drain), 0) && globaltimer_ns() - t0 < p.timeout_ns) {
        }
      }
      __syncwarp();
    } else if (warp >= 4) {
      // ---- correction (lazy O rescale) + epilogue: threads (half h, r) own
      // output columns [256h, 256h + 256) of row r
      const int r = (warp & 3) * 32 + lane;
      const int half = (warp - 4) >> 2;
      const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
      const uint32_t tcols = tmem + lane_base + half * 256;
      const bool real = g * kRows + r < p.R;
      const float* scale_buf = reinterpret_cast<const float*>(data + C::kRefOff);
      const uint32_t ml_remote = mapa(smem_u32(data + C::kMlOff), partner);
      const uint32_t mlempty_remote = mapa(smem_u32(&ctrl->ml_empty), partner);
      UnitIter it;
      it.init(p, cid);
      Unit u;
      uint32_t j = 0, un = 0, nreq = 0;
      bool ok = true;
      int why = 0;
      while (ok && it.next(u)) {
        // serve this unit's rescale requests until its last PV has landed
        // (a pending request holds back a PV of the unit, so o_full cannot
        // complete while one is pending; the next unit's first PV waits for
        // this unit's epilogue)
        const uint64_t t_unit = globaltimer_ns();
        while (true) {
          bool req = false, done = false;
          while (true) {
            req = mbar_try_wait(smem_u32(&ctrl->resc_req), nreq & 1);
            done = !req && mbar_try_wait(smem_u32(&ctrl->o_full), un & 1);
            if (__any_sync(0xffffffffu, req || done)) break;
            if (*abort || globaltimer_ns() - t_unit > p.timeout_ns) break;
            __nanosleep(32);
          }
          req = __any_sync(0xffffffffu, req);
          done = !req && __any_sync(0xffffffffu, done);
          if (!req && !done) {
            ok = false;
            why = kWaitOFull;
            break;
          }
          if (done) break;
          // page jr raised some rows' references: O *= 2^(old - new) once
          // PV(jr - 1), the last one issued, has landed
          const uint32_t jr = *reinterpret_cast<volatile uint32_t*>(&ctrl->resc_page);
          const uint32_t np = static_cast<uint32_t>(ps.n);
          if (r == 0 && half == 0) MLA_TRACE_POINT(1, 4, jr);
          const float a = real ? scale_buf[(jr % np) * ps.arows + r] : 1.f;
          if (!mbar_wait_warp<false, true>(smem_u32(&ctrl->p_empty[(jr - 1) % np]), ((jr - 1) / np) & 1, abort,
                                           p.timeout_ns)) {
            ok = false;
            why = kWaitPvPrev;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, a != 1.f)) {
            for (int c = 0; c < 256; c += 16) {
              uint32_t v[16];
              tmem_ld16(tcols + c, v);
              tmem_wait_ld_tie(v);
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * a);
              tmem_st16(tcols + c, v);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctrl->resc_done));
          if (r == 0 && half == 0) MLA_TRACE_POINT(1, 5, jr);
          ++nreq;
        }
        if (!ok) break;
        j += static_cast<uint32_t>(u.p1 - u.p0);
        // epilogue for this unit
        if (r == 0 && half == 0) MLA_TRACE_POINT(1, 13, un);
        if (r == 0 && half == 0) MLA_TRACE_POINT(1, 14, un);
        if (!mbar_wait_warp<true, true>(smem_u32(&ctrl->ml_full), un & 1, abort, p.timeout_ns)) {
          ok = false;
          why = kWaitMlFull;
          break;
        }
        tc_fence_after();
        // the two softmax groups' (frame, partial sum), brought to O's frame:
        // references never fall within a unit, so O ends in the frame of the
        // last page's reference, the higher of the two groups' last ones
        const float m0 = __uint_as_float(ld_cluster_u32(ml_remote + 16 * r));
        const float l0 = __uint_as_float(ld_cluster_u32(ml_remote + 16 * r + 4));
        const float m1 = __uint_as_float(ld_cluster_u32(ml_remote + 16 * r + 8));
        const float l1 = __uint_as_float(ld_cluster_u32(ml_remote + 16 * r + 12));
        const float m_log2 = fmaxf(m0, m1);
        const float l = l0 * ex2_approx(m0 - m_log2) + l1 * ex2_approx(m1 - m_log2);
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mlempty_remote);
        if (r == 0 && half == 0) MLA_TRACE_POINT(1, 6, un);
        store_row<kF8>(p, u, g, r, half, tmem + lane_base, m_log2, l);
        if (r == 0 && half == 0) MLA_TRACE_POINT(1, 7, un);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctrl->o_empty));
        ++un;
      }
      if (!ok && lane == 0) raise_timeout(p, ctrl, partner, why, j);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
#ifdef MLA_TRACE
  if (threadIdx.x == 0 && clus < 1024) g_mla_cluster_times[clus][1 + (rank & 1)] = globaltimer_ns();
#endif
  if (warp == 2) tmem_dealloc(tmem, 512);
  cluster_sync();
}

// ---------------------------------------------------------------- K2
// Merges the fp32 partials of every request cut by a slice boundary:
// lse = log sum_s exp(lse_s), out = sum_s exp(lse_s - lse) * out_s.

// 128 threads (4 warps, one query row each) and few registers per thread,
// so that the whole grid is resident at once when the attention kernel ends
// (with 256-thread blocks of ~100 registers only two fit per SM, and a Kimi
// batch's combine ran in three and a half waves).
constexpr int kCombineWarps = 4;
constexpr int kCombineBlocksPerSm = 7;  // 72 registers: seven 128-thread blocks per SM's 64K
constexpr int kCombineChunks = 3;  // 32 clusters each: requests over up to 96 slices take the lane-parallel path

// kParts blocks share each quad of rows, block z % kParts merging the
// z-th of kParts equal column ranges: a batch of few requests gets more
// blocks, each with more partial rows in flight per warp.
template <int kParts>
__global__ void __launch_bounds__(kCombineWarps * 32, kCombineBlocksPerSm) mla_combine_kernel(Params p) {
  static_assert(kParts == 1 || kParts == 2 || kParts == 4, "a row's 128 float4s split evenly over the lanes");
  constexpr int kV = 4 / kParts;    // float4s of a row per lane
  constexpr int kFly = 2 * kParts;  // partial rows in flight in the long walk
  // block x: entry x of the schedule's list of requests cut into pieces,
  // row block y, rows 4(z / kParts) .. + 3 (one warp each).  The schedule
  // kernel ended before the attention kernel began, so its list is read
  // before waiting for the attention kernel (through L2: an earlier call's
  // list may sit in this SM's L1); blocks past the list's end leave at
  // once, except block 0: it leaves only after the attention kernel has
  // completed, so that this grid completes after every earlier kernel of the
  // call even when nothing was cut (a kernel launched after the call as a
  // programmatic dependent then sees all of its output after its own wait).
  const bool block0 = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
  // the lse of the top-k lists without a valid pick (their decode saw one
  // all-zero key: out = 0 exactly), after the attention kernel wrote theirs
  auto empty_lists = [&]() {  // one list per thread: a flag load, then its H stores if set
    if (!p.topk_empty) return;
    for (int bq = threadIdx.x; bq < p.B; bq += blockDim.x) {
      if (!p.topk_empty[bq]) continue;
      float* l = p.lse + static_cast<int64_t>(bq) * p.H;
      for (int h = 0; h < p.H; ++h) l[h] = -INFINITY;
    }
  };
  const int nsplit = __ldcg(p.splits);
  if (static_cast<int>(blockIdx.x) >= nsplit) {
    if (block0) {
      griddep_wait();
      empty_lists();
    }
    return;
  }
  uint32_t ent[8];
  ldcg_v8(p.splits + 8 * (1 + static_cast<int64_t>(blockIdx.x)), ent);
  griddep_wait();  // the attention kernel's partials are complete
  if (block0) empty_lists();
#ifdef MLA_TRACE
  if (threadIdx.x == 0) atomicMin(&g_mla_kernel_times[2], globaltimer_ns());
  struct Exit {  // every warp stamps its exit (warps leave at different points)
    __device__ ~Exit() {
      if ((threadIdx.x & 31) == 0) atomicMax(&g_mla_kernel_times[3], globaltimer_ns());
    }
  } exit_stamp;
#endif
  MLA_COMBINE_STAMP(0);
  const int b = static_cast<int>(ent[0]), g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = static_cast<int>(blockIdx.z) % kParts;
  const int r = (static_cast<int>(blockIdx.z) / kParts) * kCombineWarps + warp;
  const int rr = g * kRows + r;
  if (rr >= p.R) return;
  const int col = lane + 32 * kV * part;  // this lane's float4s of a row: col, col + 32, ...
  const int n = static_cast<int>(ent[1]);  // pieces; ent[2 + k]: the slot of piece k
  MLA_COMBINE_STAMP(1);
  float4 acc[kV];
#pragma unroll
  for (int k = 0; k < kV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float base, z;
  auto prow_of = [&](int slot) { return (static_cast<int64_t>(slot) * p.G + g) * kRows + r; };
  auto load = [&](int64_t prow, float4 (&v)[kV]) {
    const float4* src = reinterpret_cast<const float4*>(p.o_part + prow * kDL);
#pragma unroll
    for (int q = 0; q < kV; ++q) v[q] = src[col + 32 * q];
  };
  auto add = [&](float w, const float4 (&v)[kV]) {
#pragma unroll
    for (int q = 0; q < kV; ++q) {
      acc[q].x += w * v[q].x; acc[q].y += w * v[q].y; acc[q].z += w * v[q].z; acc[q].w += w * v[q].w;
    }
  };
  if (n == 2) {
    // the common case: both pieces' lse and partial rows in flight at once
    const int64_t p0 = prow_of(static_cast<int>(ent[2])), p1 = prow_of(static_cast<int>(ent[3]));
    const float l0 = p.lse_part[p0], l1 = p.lse_part[p1];
    float4 v0[kV], v1[kV];
    load(p0, v0);
    load(p1, v1);
    const float mx = fmaxf(l0, l1);
    base = (mx == -INFINITY) ? 0.f : mx;
#ifdef MLA_TRACE
    if (v0[0].x == 12345.f && v1[0].x == 12345.f) base += 0.f;  // keeps the loads before the stamp
#endif
    MLA_COMBINE_STAMP(2);
    const float w0 = __expf(l0 - base), w1 = __expf(l1 - base);
    z = w0 + w1;
    if (w0 != 0.f) add(w0 / z, v0);
    if (w1 != 0.f) add(w1 / z, v1);
  } else if (n <= 6) {
    // the record's slots: all lse first, then the partial rows one by one
    float ls[6];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < 6; ++k) {
      ls[k] = k < n ? p.lse_part[prow_of(static_cast<int>(ent[2 + k]))] : -INFINITY;
      mx = fmaxf(mx, ls[k]);
    }
    base = (mx == -INFINITY) ? 0.f : mx;
    z = 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) z += k < n ? __expf(ls[k] - base) : 0.f;
#pragma unroll
    for (int k = 0; k < 6; ++k) {  // unrolled: the entry and ls are indexed statically (registers)
      if (k >= n) break;
      const float w = __expf(ls[k] - base) / z;
      if (w == 0.f) continue;
      float4 v[kV];
      load(prow_of(static_cast<int>(ent[2 + k])), v);
      add(w, v);
    }
  } else if (p.rrange[2 * b + 1] - p.rrange[2 * b] < 32 * kCombineChunks) {
    // more pieces (a request spanning many slices).  Lane l takes the
    // clusters clo + l, clo + l + 32, ... whose slice meets the request (an
    // empty slice holds no piece: weight 0), loads their lse at once and the
    // warp reduces max and sum; then the warp walks the clusters in order,
    // weights and slots broadcast, kFly partial rows in flight.  (A walk
    // with a load per piece and per pass took ~50 us for one request over
    // 76 slices.)
    const int clo = p.rrange[2 * b], chi = p.rrange[2 * b + 1];
    int slv[kCombineChunks];
    float lsv[kCombineChunks];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kCombineChunks; ++k) {
      const int c = clo + 32 * k + lane;
      slv[k] = 0;
      lsv[k] = -INFINITY;
      if (c <= chi && p.cinfo[3 * c] != p.cinfo[3 * c + 1]) {
        slv[k] = 2 * c + (b != p.cinfo[3 * c + 2] ? 1 : 0);
        lsv[k] = p.lse_part[prow_of(slv[k])];
      }
      mx = fmaxf(mx, lsv[k]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    base = (mx == -INFINITY) ? 0.f : mx;
    float wv[kCombineChunks];
    z = 0.f;
#pragma unroll
    for (int k = 0; k < kCombineChunks; ++k) {
      wv[k] = lsv[k] == -INFINITY ? 0.f : __expf(lsv[k] - base);
      z += wv[k];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
#pragma unroll
    for (int k = 0; k < kCombineChunks; ++k) wv[k] /= z;
#pragma unroll
    for (int k = 0; k < kCombineChunks; ++k) {
      if (clo + 32 * k > chi) break;
#pragma unroll 1
      for (int j = 0; j < 32; j += kFly) {
        float wf[kFly];
        int sf[kFly];
#pragma unroll
        for (int q = 0; q < kFly; ++q) {
          wf[q] = __shfl_sync(0xffffffffu, wv[k], j + q);
          sf[q] = __shfl_sync(0xffffffffu, slv[k], j + q);
        }
        float4 v[kFly][kV];
#pragma unroll
        for (int q = 0; q < kFly; ++q) {
          const float4* src = reinterpret_cast<const float4*>(p.o_part + prow_of(sf[q]) * kDL);
#pragma unroll
          for (int e = 0; e < kV; ++e) v[q][e] = wf[q] != 0.f ? src[col + 32 * e] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < kFly; ++q)
          if (wf[q] != 0.f) add(wf[q], v[q]);
      }
    }
  } else {
    // more clusters than the lanes take at once: walk them one by one
    const int clo = p.rrange[2 * b], chi = p.rrange[2 * b + 1];
    float mx = -INFINITY;
    for (int c = clo; c <= chi; ++c) {
      if (p.cinfo[3 * c] == p.cinfo[3 * c + 1]) continue;
      mx = fmaxf(mx, p.lse_part[prow_of(2 * c + (b != p.cinfo[3 * c + 2] ? 1 : 0))]);
    }
    base = (mx == -INFINITY) ? 0.f : mx;
    z = 0.f;
    for (int c = clo; c <= chi; ++c) {
      if (p.cinfo[3 * c] == p.cinfo[3 * c + 1]) continue;
      z += __expf(p.lse_part[prow_of(2 * c + (b != p.cinfo[3 * c + 2] ? 1 : 0))] - base);
    }
    for (int c = clo; c <= chi; ++c) {
      if (p.cinfo[3 * c] == p.cinfo[3 * c + 1]) continue;
      const int64_t prow = prow_of(2 * c + (b != p.cinfo[3 * c + 2] ? 1 : 0));
      const float w = __expf(p.lse_part[prow] - base) / z;
      if (w == 0.f) continue;
      float4 v[kV];
      load(prow, v);
      add(w, v);
    }
  }
  const int i = rr / p.H, h = rr % p.H;
  const int64_t orow = (static_cast<int64_t>(b) * p.Q + i) * p.H + h;
  if (p.out_f32) {
    float4* dstf = reinterpret_cast<float4*>(p.out + orow * kDL * 4);
#pragma unroll
    for (int k = 0; k < kV; ++k) dstf[col + 32 * k] = acc[k];
    if (lane == 0 && part == 0) p.lse[orow] = base + __logf(z);
    return;
  }
  uint2* dst = reinterpret_cast<uint2*>(p.out + orow * kDL * 2);
#pragma unroll
  for (int k = 0; k < kV; ++k) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[k].x, acc[k].y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[k].z, acc[k].w);
    dst[col + 32 * k] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
  if (lane == 0 && part == 0) p.lse[orow] = base + __logf(z);
  MLA_COMBINE_STAMP(3);
}

// ------------------------------------------------------ gather test hook
struct GatherParams {
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int64_t* row_offsets;
  uint8_t* rows_out;
  int32_t* status;
  int32_t B, num_pages, max_pages, pt_stride;
  uint64_t timeout_ns;
};

template <bool kF8>
__global__ void __launch_bounds__(128) mla_gather_kernel(const __grid_constant__ GatherParams gp,
                                                         const __grid_constant__ CUtensorMap tm_s,
                                                         const __grid_constant__ CUtensorMap tm_pe) {
  using C = Cfg<kF8>;
  extern __shared__ uint8_t smem_raw[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw);
  int* abort_flag = reinterpret_cast<int*>(smem_raw + 8);
  uint8_t* page = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 64 + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int pg = blockIdx.x, b = blockIdx.y;
  const int L = clamp_len(gp.seq_lens[b], gp.max_pages);
  const int np = (L + kPage - 1) / kPage;
  if (pg >= np) return;
  int32_t pid = gp.page_table[static_cast<int64_t>(b) * gp.pt_stride + pg];
  if (pid < 0 || pid >= gp.num_pages) {
    if (threadIdx.x == 0) atomicOr(gp.status, MLA_DEV_BAD_PAGE_ID);
    pid = 0;
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(bar), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // exactly the loads of the decode kernel's S CTA
    mbar_expect_tx(smem_u32(bar), C::kSlotS);
    tma_load_3d(smem_u32(page), &tm_s, 0, pid * kPage, 0, smem_u32(bar));
    if constexpr (kF8) tma_load_2d(smem_u32(page + C::kNBoxLat * C::kBox), &tm_pe, kDL, pid * kPage, smem_u32(bar));
  }
  if (!mbar_wait(smem_u32(bar), 0, abort_flag, gp.timeout_ns)) {
    if (threadIdx.x == 0) atomicOr(gp.status, MLA_DEV_TIMEOUT);
    // the copy may still be in flight: wait for it (bounded) before leaving
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(smem_u32(bar), 0) && globaltimer_ns() - t0 < gp.timeout_ns) {
    }
    return;
  }
  const int valid = L - pg * kPage < kPage ? L - pg * kPage : kPage;
  const int row_bytes = 576 * C::kEsz;
  uint8_t* dst0 = gp.rows_out + (gp.row_offsets[b] + static_cast<int64_t>(pg) * kPage) * row_bytes;
  // 16-byte chunks: c_kv boxes have 8 chunks per token row, the k_pe box 8 (bf16) or 4 (e4m3)
  const int lat_chunks = C::kNBoxLat * 8;
  const int pe_chunks = kF8 ? 4 : 8;
  const int per_row = lat_chunks + pe_chunks;
  for (int idx = threadIdx.x; idx < valid * per_row; idx += blockDim.x) {
    const int t = idx / per_row, c = idx % per_row;
    uint4 v;
    if (c < lat_chunks) {
      const int box = c / 8, ch = c % 8;
      v = *reinterpret_cast<const uint4*>(page + box * C::kBox + t * 128 + ((ch ^ (t & 7)) << 4));
    } else {
      const int ch = c - lat_chunks;
      if constexpr (kF8)
        v = *reinterpret_cast<const uint4*>(page + C::kNBoxLat * C::kBox + t * 64 + ((ch ^ ((t >> 1) & 3)) << 4));
      else
        v = *reinterpret_cast<const uint4*>(page + C::kNBoxLat * C::kBox + t * 128 + ((ch ^ (t & 7)) << 4));
    }
    *reinterpret_cast<uint4*>(dst0 + static_cast<int64_t>(t) * row_bytes + c * 16) = v;
  }
}

// ---------------------------------------------- bounded-wait self-test
__global__ void mla_wait_selftest_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up after limit_ns
  if (!mbar_wait(smem_u32(&bar), 0, &abort_flag, limit_ns)) {
    if (threadIdx.x == 0) atomicOr(status, MLA_DEV_TIMEOUT);
  }
}

}  // namespace mla
