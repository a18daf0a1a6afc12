// Varlen paged attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// with TMA-gathered K/V: step 2 of the paged-kernel contract ("Attention
// Backends", section "What 'paged attention' requires of a kernel") computed
// as O = softmax(Q K^T * scale + M) V ("Chapter 1: attention backends",
// section 2.1) with the FlashAttention tiling and online softmax of section
// 4.1.
//
// CTA = (256 packed rows as two Q tiles of 128, kv head, request); a packed
// row is one (query row, q head of the kv group) pair, so the Hq/Hkv heads
// sharing a kv head share every K/V tile.  Warp roles (384 threads):
//   warp 0     MMA issue (one thread; with MLA keys warp 2 too, one thread
//              per Q tile): S_x(j) = Q_x K(j)^T, then O_x += P_x(j) V(j)
//              with the A operand (P) read from TMEM;
//   warp 1     K/V producer: per 16-token piece of a cache block one TMA box
//              per 64-column half of K and one box for both halves of V,
//              through the block table;
//   warps 2-3  idle otherwise (they complete the first warpgroup, which
//              hands its registers to the softmax warpgroups);
//   warps 4-7 / 8-11  two softmax warpgroups, one per Q tile: thread t of a
//              group owns row t of its tile = TMEM lane t.  Per 128-token K/V
//              tile it reads its S row from TMEM, masks (causal,
//              bottom-right), runs the online softmax in the log2 domain and
//              writes its P row (bf16, two per 32-bit column) back into TMEM
//              over the S row it came from.
// The MMA and producer warps have the lowest warp ids: each shares its
// scheduler with two busy softmax warps, and the low ids keep them from being
// starved of issue slots.
// The two Q tiles interleave on the tensor core (PV_0(j), S_0(j+1), PV_1(j),
// S_1(j+1), ... from one thread; with two issuers each tile's PV_x(j) and
// S_x(j+1) as soon as P_x(j) is written), so each softmax warpgroup works on
// one tile while the MMAs of the other proceed.  The tensor pipe runs in
// issue order and S_x(j) follows PV_x(j-1) from the same thread, so once
// S_x(j) has landed PV_x(j-1) has too: the softmax may rescale O_x (TMEM
// load, scale, store) without another wait; it does so only when a row's
// running max grows by more than 2^8 (P keeps the older reference max
// otherwise, which keeps O / l exact).
//
// Shared memory (128-byte swizzled, 1024-byte aligned atoms):
//   Q    2 tiles x [DK/64 halves][128 rows][128 B]
//   K    2 stages x [DK/64 halves][BN tokens][128 B]
//   V    VST stages x [BN/16 pieces][DV/64 halves][16 tokens][128 B] (the MLA
//        workspaces: [DV/64 halves][BN tokens][128 B])
// (DK = DV = d and BN = 128 for the standard pool; DK = 192, DV = 128 and
// BN = 64 for the MLA prefill, whose queries and keys are [nope | rope].)
// TMEM (512 columns): S_0/P_0 at 0, S_1/P_1 at 128, O_0 at 256, O_1 at 384.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"
#include "tc_common.cuh"

namespace pa {

// DK: width of queries and keys; DV: width of values and outputs; BN: tokens
// per K/V tile; VST: V stages (2, or 1 where two do not fit).
template <int DK, int DV, int BN, int VST = 2>
struct TcCfg {
  static constexpr int kVStages = VST;
  static constexpr int kBM = 128;                     // rows per Q tile
  static constexpr int kRows = 2 * kBM;               // packed rows per CTA
  static constexpr int kBN = BN;                      // tokens per K/V tile
  static constexpr int kHalvesK = DK / 64;            // 128-byte column groups of a key row
  static constexpr int kHalvesV = DV / 64;            // ... of a value row
  static constexpr int kQBytes = kBM * DK * 2;        // one Q tile
  static constexpr int kKBytes = kBN * DK * 2;        // one K tile
  static constexpr int kVBytes = kBN * DV * 2;        // one V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + 2 * kKBytes;
  static constexpr int kOffBar = kOffV + VST * kVBytes;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;   // barriers + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 384;
  // Registers per thread: the softmax warpgroups 1-2 raise theirs,
  // warpgroup 0 (MMA issue, producer, two idle warps) lowers its own.  The launch must
  // hold at least 256 * kRegSoftmax + 128 * kRegOther registers.
  static constexpr uint32_t kRegSoftmax = 216;
  static constexpr uint32_t kRegOther = 56;
  static constexpr int kPieceBytes = 16 * 128;        // one TMA box: 16 rows x 128 B
  __host__ __device__ static constexpr uint32_t col_s(int x) { return 128u * x; }
  __host__ __device__ static constexpr uint32_t col_o(int x) { return 256u + 128u * x; }
};

// Byte offset of 16-byte chunk `c` (0..7) of row `r` in a 128-byte swizzled
// [rows][128 B] region.
__device__ __forceinline__ uint32_t sw128(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Barriers; pairs are indexed by stage (j & 1) or by Q tile x.
enum TcBar {
  kQFull = 0,
  kKFull = 1,
  kKEmpty = 3,
  kVFull = 5,
  kVEmpty = 7,
  kSFull = 9,    // [x]
  kPLo = 11,     // [x] P columns of tokens 0-63 written
  kPHi = 13,     // [x] P columns of tokens 64-127 written
  kODone = 15,   // [x]
  kFinal = 17,
  kNumBars = 18
};
// Arguments of one varlen launch.  The plain call fills the first block; the
// rest serve split-KV partials and the two passes of cascade attention.
struct VarlenArgs {
  const __nv_bfloat16* q;
  const int32_t* block_table;
  const int32_t* qsl;
  const int32_t* seq_lens;
  int max_blocks;   // row stride of block_table
  int Hq, Hkv, bs, num_blocks;
  float scale_log2;
  int causal;
  int window;       // > 0: sliding window (causal), row at p sees p - window < p' <= p
  __nv_bfloat16* out;
  float* lse;
  int* err;
  int table_col0;   // a request's blocks start at this column of its row
  int seq_off;      // tokens dropped from the front of every request (seq_lens[i] - seq_off)
  int virt_total_q; // > 0: one request made of query rows [0, virt_total_q) ...
  int virt_seq;     // ... over virt_seq tokens of table row 0 (qsl, seq_lens unused)
  float* ws;        // non-null: partial output, [rows][Hq][ws_slots][DV + 1] fp32
  int ws_slots, ws_slot0;
  int kv_splits;    // context cut into kv_splits pieces of kv_chunk (a multiple of the tile)
  int kv_chunk;
  int mla_s_max;    // MLA mode: token rows per request in the expanded workspaces
};

// After the barriers: the TMEM base address (4 B, padded to 8), the abort
// flag (4 B, padded to 8) and a ring of 4 tile descriptors (4 B each).
constexpr int kPieceRing = 4;

#ifdef PA_TEST_HOOKS
// Test builds only: the producer of the CTA whose linear block index is
// g_test_skip.x issues no copies (and no byte count) for K/V tile
// g_test_skip.y, so the waits on that tile's barriers can only end at their
// poll limit.  Set by pa_test_skip_tile_loads; {-1, -1} = off.
__device__ int2 g_test_skip = {-1, -1};
#endif

// EXT = false compiles the plain call (no window, split, offsets, virtual
// request or partial output: those fields are ignored).
// MLA = true: keys and values come from the contiguous expanded workspaces
// of the MLA prefill (k_map over [N * s_max][H][DK], v_map over
// [N * s_max][H][DV]) instead of the paged pool; no block table.
template <int DK, int DV, int BN, int VST, bool EXT, bool MLA>
__global__ void __launch_bounds__(384, 1)
varlen_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap v_map,
                 const __grid_constant__ VarlenArgs a) {
  using C = TcCfg<DK, DV, BN, VST>;
  // Standard pool: a V piece (16 tokens, both halves) is one TMA box, laid
  // out [half][16 tokens][128 B]; TMA issue, not bandwidth, is what the
  // producer spends its time on, so V takes half the boxes of K.
  constexpr bool kVm = !MLA;
  constexpr uint32_t kVPiece = C::kHalvesV * C::kPieceBytes;
  // MMA issue by one thread per Q tile (measured faster for the MLA shape:
  // 192-wide keys, one V stage) or by one thread for both (faster for the
  // standard pool).
  constexpr bool kTwoIssuers = MLA;
  constexpr uint32_t kIssuers = kTwoIssuers ? 2 : 1;
  const __nv_bfloat16* __restrict__ q = a.q;
  const int32_t* __restrict__ block_table = a.block_table;
  const int Hq = a.Hq, Hkv = a.Hkv, bs = a.bs, num_blocks = a.num_blocks;
  const int causal = a.causal, window = EXT ? a.window : 0;
  const int table_col0 = EXT ? a.table_col0 : 0, seq_off = EXT ? a.seq_off : 0;
  const int kv_splits = EXT ? a.kv_splits : 1;
  float* const ws = EXT ? a.ws : nullptr;
  const float scale_log2 = a.scale_log2;
  __nv_bfloat16* __restrict__ out = a.out;
  float* __restrict__ lse = a.lse;
  int* err = a.err;
  // Usable table columns of a request's row (the row starts at column
  // table_col0 of a max_blocks-wide table).
  const int max_blocks = a.max_blocks - table_col0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);

  const int i = blockIdx.z, kvh = blockIdx.y;
  // blockIdx.x = split * q_tiles + (q tile counted from the last).
  const int q_tiles = static_cast<int>(gridDim.x) / kv_splits;
  const int split = EXT ? static_cast<int>(blockIdx.x) / q_tiles : 0;
  const int qt = EXT ? q_tiles - 1 - static_cast<int>(blockIdx.x) % q_tiles
                     : static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x);  // heavy tiles first
  const int grp = Hq / Hkv;
  // A virtual request (virt_total_q > 0) is every query row of the call
  // against one fixed context of virt_seq tokens read through table row 0.
  const bool virt = EXT && a.virt_total_q > 0;
  const int q0 = virt ? 0 : a.qsl[i];
  const int qlen = virt ? a.virt_total_q : a.qsl[i + 1] - q0;
  const int rows_total = qlen * grp;
  if (qt * C::kRows >= rows_total) return;      // nothing to do
  const int row0 = qt * C::kRows;               // this CTA's rows (may all be past the end)
  const int seq = virt ? a.virt_seq : max(0, a.seq_lens[i] - seq_off);
  const int ctx = seq - qlen;
  if (EXT && !virt && causal && ctx < 0 && seq_off > 0 && threadIdx.x == 0 && blockIdx.x == 0 &&
      blockIdx.y == 0)
    record_error(err, PA_DEVERR_LENGTH);   // queries inside the skipped prefix
  const int last_row = min((qt + 1) * C::kRows, rows_total) - 1;   // this CTA's last row
  int kv_end = causal ? ctx + last_row / grp + 1 : seq;
  kv_end = max(0, min(kv_end, seq));
  // Sliding window (causal only): the CTA's first row sees nothing
  // before ctx + q_first + 1 - window, so the tiles start at that position
  // rounded down to a tile; later rows mask their own lower bound.
  int tbase = 0;
  if (window > 0) {
    const int q_first = min(qt * C::kRows, rows_total - 1) / grp;
    tbase = max(0, ctx + q_first + 1 - window) / C::kBN * C::kBN;
  }
  // KV split (a multiple of the tile): this CTA covers [split * kv_chunk,
  // (split + 1) * kv_chunk) of the context, the last split to its end.
  if (kv_splits > 1) {
    const long long s0 = static_cast<long long>(split) * a.kv_chunk;
    tbase = static_cast<int>(max(static_cast<long long>(tbase), s0));
    if (split < kv_splits - 1) kv_end = static_cast<int>(min(static_cast<long long>(kv_end), s0 + a.kv_chunk));
  }
  tbase = min(tbase, kv_end);
  const int ntiles = (kv_end - tbase + C::kBN - 1) / C::kBN;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* table =
      block_table + static_cast<int64_t>(virt ? 0 : i) * a.max_blocks + table_col0;

  const uint32_t bars = sbase + C::kOffBar;
  auto BAR = [&](int k) { return bars + 8u * static_cast<uint32_t>(k); };
  const uint32_t tmem_slot = bars + 8u * kNumBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 8 * kNumBars + 8);
  // Ring of loaded-piece masks: the producer writes (j << 8) | mask for tile
  // j into slot j % kPieceRing before it issues K(j); the softmax reads it
  // once S(j) has landed.  The tag makes the slot self-validating.
  volatile uint32_t* piece_ring =
      reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kNumBars + 16);

  if (threadIdx.x == 0) {
    tc::mbar_init(BAR(kQFull), C::kRows);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(BAR(kKFull + b), 1);
      // Released by every issuing thread.
      tc::mbar_init(BAR(kKEmpty + b), kIssuers);
      tc::mbar_init(BAR(kVFull + b), 1);
      tc::mbar_init(BAR(kVEmpty + b), kIssuers);
      tc::mbar_init(BAR(kSFull + b), 1);
      tc::mbar_init(BAR(kPLo + b), C::kBM);
      tc::mbar_init(BAR(kPHi + b), C::kBM);
      tc::mbar_init(BAR(kODone + b), 1);
    }
    tc::mbar_init(BAR(kFinal), kIssuers);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) tc::tmem_alloc(tmem_slot, C::kTmemCols);
  tc::tc_fence_before();
  // The launch is a cluster of one CTA, so the cluster barrier is a split
  // barrier of this CTA: every thread arrives now and waits just before its
  // first use of TMEM, and the Q rows and the first block ids are fetched
  // while the TMEM allocation completes.
  tc::cluster_arrive();
  auto tmem_base = [&]() {
    return *reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kNumBars);
  };
  auto release = [&](uint32_t bar) { tc::mma_commit(bar); };   // frees a K/V stage
  auto fail = [&]() {
    record_error(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp >= 4)
    tc::reg_alloc<C::kRegSoftmax>();
  else
    tc::reg_dealloc<C::kRegOther>();

  if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int x = (warp >> 2) - 1;           // Q tile of this warpgroup
    const int t = threadIdx.x & 127;         // row within the tile = TMEM lane
    const int pr = row0 + x * C::kBM + t;
    const bool valid = pr < rows_total;
    const int qi = valid ? pr / grp : 0;
    const int hh = valid ? pr % grp : 0;
    const int64_t qrow = static_cast<int64_t>(q0 + qi) * Hq + kvh * grp + hh;
    const int64_t qoff = qrow * DK;
    int lim = valid ? (causal ? ctx + qi + 1 : seq) : 0;
    lim = max(0, min(lim, seq));
    const int lo = window > 0 ? max(0, lim - window) : 0;   // first visible position
    {
      const uint4* src = reinterpret_cast<const uint4*>(q + qoff);
      const uint32_t qb = sbase + C::kOffQ + x * C::kQBytes;
#pragma unroll
      for (int c = 0; c < DK / 8; ++c) {
        uint4 v = valid ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
        const uint32_t dst = qb + (c >> 3) * (C::kBM * 128) + sw128(t, c & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w)
                     : "memory");
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(BAR(kQFull));
    }
    tc::cluster_wait();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base();
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_base + C::col_s(x), to = tmem + lane_base + C::col_o(x);
    // TMEM loads and stores are warp-collective: every decision to skip or
    // stop is taken for the whole warp.
    auto wait_warp = [&](uint32_t b, uint32_t parity) -> bool {
      const bool w = __all_sync(0xffffffffu, tc::mbar_wait(b, parity));
      if (!w) fail();
      return w;
    };
    // l: the row's sum of weights (for the LSE); lr: the same weights rounded
    // to bf16, as PV multiplies them (the output's divisor, so that a
    // dominant token's value is not scaled by the rounding of its weight).
    float m_used = -CUDART_INF_F, l = 0.f, lr = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int tok0 = tbase + j * C::kBN;
      if (!wait_warp(BAR(kSFull + x), j & 1)) break;
      tc::tc_fence_after();
      // Loaded pieces of this tile, from the producer's ring (written before
      // K(j) was issued, so normally visible at the first read).
      uint32_t vm;
      {
        const uint32_t tag = static_cast<uint32_t>(j) << 8;
        uint32_t w = piece_ring[j % kPieceRing];
        for (int n = 0; (w & ~0xffu) != tag && n < tc::kWaitPolls; ++n) w = piece_ring[j % kPieceRing];
        if (!__all_sync(0xffffffffu, (w & ~0xffu) == tag)) {
          fail();
          break;
        }
        vm = w & 0xffu;
      }
      float s[C::kBN];
      {
        uint32_t r[C::kBN / 32][32];
#pragma unroll
        for (int c = 0; c < C::kBN / 32; ++c) tc::tmem_ld32(ts + c * 32, r[c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < C::kBN / 32; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) s[c * 32 + e] = __uint_as_float(r[c][e]);
      }
      // Mask only where some column is not visible (the diagonal tile, the
      // end of the sequence, the window's start, an unloaded piece).
      if (!(tok0 + C::kBN <= lim && tok0 >= lo && vm == (1u << (C::kBN / 16)) - 1u)) {
#pragma unroll
        for (int col = 0; col < C::kBN; ++col) {
          const bool vis = (tok0 + col < lim) && (tok0 + col >= lo) && ((vm >> (col >> 4)) & 1u);
          s[col] = vis ? s[col] : -CUDART_INF_F;
        }
      }
      float mx;
      {
        // Eight independent chains of 3-input maxima, then their maximum.
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(s[k], s[8 + k]);
#pragma unroll
        for (int col = 16; col < C::kBN; col += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = max3(m8[k], s[col + k], s[col + 8 + k]);
        mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        mx *= scale_log2;
      }
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;
      const float alpha = need ? ex2(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
      // S_x(j) has landed, hence PV_x(j-1) too: O_x may be rescaled now.
      if (__any_sync(0xffffffffu, need) && j > 0) {
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(to + c * 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tc::tmem_st32(to + c * 32, r);
        }
      }
      // V rows that must contribute nothing: past seq_len (stale or unset
      // cache contents) or in pieces that were not loaded.  Zeroed once the
      // tile's V has landed (one row per thread) by both warpgroups, each
      // before it publishes its own P: PV_0(j) and PV_1(j) go out in either
      // order.  Both write zeros, so the overlap is harmless.
      {
        const int tok = tok0 + t;
        // Threads past the tile's kBN rows own no V row.
        const bool row_ok = t >= C::kBN || (tok < seq && ((vm >> (t >> 4)) & 1u));
        if (!row_ok) {
          if (!tc::mbar_wait(BAR(kVFull + j % C::kVStages), (j / C::kVStages) & 1)) fail();
          const uint32_t vbase = sbase + C::kOffV + (j % C::kVStages) * C::kVBytes;
#pragma unroll
          for (int h = 0; h < C::kHalvesV; ++h)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t dst =
                  kVm ? vbase + (t >> 4) * kVPiece + h * C::kPieceBytes + sw128(t & 15, c)
                      : vbase + h * (C::kBN * 128) + sw128(t, c);
              asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
            }
          tc::fence_proxy_async_smem();   // before this thread's P arrival
        }
      }
      // P = exp2(s * scale_log2 - m_used) as bf16 pairs over the first 64
      // columns of the S row, published in two halves (tokens 0-63, 64-127)
      // so that the first half of PV_x(j) runs while the second is computed.
      {
        // Row sums in eight partial sums, four packed pairs (and the same
        // for the rounded weights).
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c16 = 0; c16 < C::kBN / 32; ++c16) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = c16 * 16 + e;
            float x0, x1;
            ffma2(x0, x1, s[2 * c], s[2 * c + 1], scale_log2, -mu);
            const float p0 = ex2(x0);
            const float p1 = ex2(x1);
            fadd2(l8[2 * (e & 3)], l8[2 * (e & 3) + 1], p0, p1);
            pk[e] = pack_bf16(p0, p1);
            add_bf16x2_f32(r8[2 * (e & 3)], r8[2 * (e & 3) + 1], pk[e]);
          }
          tc::tmem_st16(ts + c16 * 16, pk);
          if (c16 == C::kBN / 64 - 1 || c16 == C::kBN / 32 - 1) {
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(BAR((c16 == C::kBN / 32 - 1 ? kPHi : kPLo) + x));
          }
        }
        l = l * alpha + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
        lr = lr * alpha + (((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7])));
      }
    }
    // ------------------------------------------------------------ epilogue
    bool ok = !__any_sync(0xffffffffu, *abort_flag != 0) && ntiles > 0;
    if (ok) ok = wait_warp(BAR(kODone + x), (ntiles - 1) & 1);
    tc::tc_fence_after();
    // Partial mode: the row's normalised output and LSE go, in fp32, to slot
    // ws_slot0 + split of its workspace row [ws_slots][DV + 1].
    float* wrow = ws == nullptr ? nullptr
                                : ws + (qrow * a.ws_slots + a.ws_slot0 + split) * (DV + 1);
    if (ok && wrow != nullptr) {   // warp-uniform
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(to + c * 32, r);
        tc::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int e = 0; e < 32; ++e) wrow[c * 32 + e] = __uint_as_float(r[e]) * inv;
        }
      }
      if (valid) wrow[DV] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
    } else if (wrow != nullptr) {
      if (valid) {
        for (int c = 0; c < DV; ++c) wrow[c] = 0.f;
        wrow[DV] = -CUDART_INF_F;
      }
    } else if (ok) {   // warp-uniform
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
      // A warp's store covers 32 rows (one per thread): 32-byte stores write
      // whole sectors where `out` is 32-byte aligned (rows are multiples of
      // 32 bytes), 16-byte ones otherwise.
      const bool a32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
      uint32_t* dst = reinterpret_cast<uint32_t*>(out + qrow * DV);
#pragma unroll
      for (int c2 = 0; c2 < DV / 64; ++c2) {
        uint32_t r[2][32];
        tc::tmem_ld32(to + c2 * 64, r[0]);
        tc::tmem_ld32(to + c2 * 64 + 32, r[1]);
        tc::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w[e] = pack_bf16(__uint_as_float(r[u][v * 16 + 2 * e]) * inv,
                                 __uint_as_float(r[u][v * 16 + 2 * e + 1]) * inv);
              uint32_t* p = dst + (c2 * 2 + u) * 16 + v * 8;
              if (a32) {
                st_global_v8(p, w);
              } else {
                reinterpret_cast<uint4*>(p)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                reinterpret_cast<uint4*>(p)[1] = make_uint4(w[4], w[5], w[6], w[7]);
              }
            }
        }
      }
      if (valid && lse != nullptr)
        lse[qrow] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
    } else if (valid) {
      // Nothing visible (or an aborted CTA): o = 0, lse = -inf.
      uint4* dst = reinterpret_cast<uint4*>(out + qrow * DV);
      for (int c = 0; c < DV / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
      if (lse != nullptr) lse[qrow] = -CUDART_INF_F;
    }
  } else if (warp == 0 || (kTwoIssuers && warp == 2)) {
    // ------------------------------------------------------------ MMA issue
    tc::cluster_wait();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_base();
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, C::kBN, 0, 0);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, DV, 0, 1);
      bool ok = ntiles == 0 || tc::mbar_wait(BAR(kQFull), 0);
      if (!ok) fail();
      // S_x(j) = Q_x K(j)^T into the S columns of tile x.
      auto issue_s = [&](int xq, int j) {
        const uint32_t qs = sbase + C::kOffQ + xq * C::kQBytes;
        const uint32_t ks = sbase + C::kOffK + (j & 1) * C::kKBytes;
#pragma unroll
        for (int k = 0; k < DK / 16; ++k) {
          const uint32_t off = (k >> 2) * (C::kBM * 128) + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * (C::kBN * 128) + (k & 3) * 32;
          tc::mma_bf16_ss(tmem + C::col_s(xq), tc::smem_desc_sw128(qs + off, 16, 1024),
                          tc::smem_desc_sw128(ks + koff, 16, 1024), idesc_s, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(BAR(kSFull + xq));
      };
      // O_x += P_x(j) V(j) over the 16-token steps [k0, k0 + 4); P_x is read
      // from TMEM, 8 columns (16 bf16) per step.
      auto issue_pv = [&](int xq, int j, int k0) {
        const uint32_t vs = sbase + C::kOffV + (j % C::kVStages) * C::kVBytes;
#pragma unroll
        for (int k = k0; k < k0 + C::kBN / 32; ++k)
          tc::mma_bf16_ts(tmem + C::col_o(xq), tmem + C::col_s(xq) + k * 8,
                          kVm ? tc::smem_desc_sw128(vs + k * kVPiece, C::kPieceBytes, 1024)
                              : tc::smem_desc_sw128(vs + k * 16 * 128, C::kBN * 128, 1024),
                          idesc_o,
                          (j > 0 || k > 0) ? 1u : 0u);
      };
      auto wait_k = [&](int j) { return tc::mbar_wait(BAR(kKFull + (j & 1)), (j >> 1) & 1); };
      if (kTwoIssuers) {
        // Each Q tile has its own issuing thread (warp 0: tile 0, warp 2:
        // tile 1).  A thread blocks while the tensor pipe's queue is full, so
        // with one thread for both tiles P_0(j+1), long written, can wait
        // behind tile 1's batch; with two, each tile's PV and next S go out
        // as soon as its own P is ready.  tcgen05.commit tracks the issuing
        // thread's own MMAs, so each thread releases the K and V stages for
        // its tile (the empty barriers count both threads).
        const int xq = warp == 0 ? 0 : 1;
        if (ok && ntiles > 0) {
          ok = wait_k(0);
          if (ok) {
            tc::tc_fence_after();
            issue_s(xq, 0);
            release(BAR(kKEmpty + 0));
          }
        }
        for (int j = 0; ok && j < ntiles; ++j) {
          if (*abort_flag) { ok = false; break; }
          const bool more = j + 1 < ntiles;
          if (!tc::mbar_wait(BAR(kVFull + j % C::kVStages), (j / C::kVStages) & 1)) { ok = false; break; }
          if (!tc::mbar_wait(BAR(kPLo + xq), j & 1)) { ok = false; break; }
          tc::tc_fence_after();
          issue_pv(xq, j, 0);
          if (!tc::mbar_wait(BAR(kPHi + xq), j & 1)) { ok = false; break; }
          tc::tc_fence_after();
          issue_pv(xq, j, C::kBN / 32);
          tc::mma_commit(BAR(kODone + xq));
          // K(j+1) only now: PV_x(j) does not need it.
          if (more && !wait_k(j + 1)) { ok = false; break; }
          tc::tc_fence_after();
          if (more) issue_s(xq, j + 1);
          release(BAR(kVEmpty + j % C::kVStages));
          if (more) release(BAR(kKEmpty + ((j + 1) & 1)));
        }
      } else {
        // One thread for both tiles: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).
        if (ok && ntiles > 0) {
          ok = wait_k(0);
          if (ok) {
            tc::tc_fence_after();
            issue_s(0, 0);
            issue_s(1, 0);
            release(BAR(kKEmpty + 0));
          }
        }
        for (int j = 0; ok && j < ntiles; ++j) {
          if (*abort_flag) { ok = false; break; }
          const bool more = j + 1 < ntiles;
          if (!tc::mbar_wait(BAR(kVFull + j % C::kVStages), (j / C::kVStages) & 1)) { ok = false; break; }
          if (more && !wait_k(j + 1)) { ok = false; break; }
          for (int xq = 0; xq < 2 && ok; ++xq) {
            if (!tc::mbar_wait(BAR(kPLo + xq), j & 1)) { ok = false; break; }
            tc::tc_fence_after();
            issue_pv(xq, j, 0);
            if (!tc::mbar_wait(BAR(kPHi + xq), j & 1)) { ok = false; break; }
            tc::tc_fence_after();
            issue_pv(xq, j, C::kBN / 32);
            tc::mma_commit(BAR(kODone + xq));
            if (more) issue_s(xq, j + 1);
          }
          if (!ok) break;
          release(BAR(kVEmpty + j % C::kVStages));
          if (more) release(BAR(kKEmpty + ((j + 1) & 1)));
        }
      }
      if (!ok && !*abort_flag) fail();
      // Everything issued has completed before TMEM is released.
      tc::mma_commit(BAR(kFinal));
      if (!tc::mbar_wait(BAR(kFinal), 0)) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ K/V producer
    // Lane p looks after the tile's 16-token piece p: its block id (loaded
    // three tiles ahead and validated only when used, so the load's latency
    // never stalls an issue) and its TMA boxes (one per 64-column half of K,
    // one for both halves of V).  The barrier expects the bytes of all loaded
    // pieces.  V(j) goes out before
    // K(j+2) (PV(j) needs it first) and reuses K(j)'s block ids.
    if (lane == 0) {
      tc::tma_prefetch_desc(&kv_map);
      tc::tma_prefetch_desc(&v_map);
    }
    const int pc = lane;
    const bool box_lane = lane < C::kBN / 16;
    const bool my_piece = box_lane;
    auto in_range = [&](int j) -> bool {
      return box_lane && j < ntiles && tbase + j * C::kBN + 16 * pc < kv_end;
    };
    auto raw_of = [&](int j) -> int {
      if (!in_range(j)) return -1;
      if (MLA) return 0;   // contiguous workspace: every in-range piece is loaded
      const int idx = (tbase + j * C::kBN + 16 * pc) / bs;
      return idx < max_blocks ? __ldg(table + idx) : -1;
    };
    // The piece's block id, -1 (not visible) or -2 (invalid id).
    auto valid_of = [&](int j, int raw) -> int {
      return !in_range(j) ? -1 : (raw >= 0 && raw < num_blocks) ? raw : -2;
    };
    auto issue = [&](int j, int blk, int which, uint32_t dst, uint32_t full) {
      const int tok0 = tbase + j * C::kBN;
      const unsigned loaded = __ballot_sync(0xffffffffu, blk >= 0);
      const unsigned bad = __ballot_sync(0xffffffffu, blk == -2);
      if (lane == 0) {
        if (bad != 0u && which == 0) record_error(err, PA_DEVERR_BLOCK_ID);
        if (which == 0) piece_ring[j % kPieceRing] = (static_cast<uint32_t>(j) << 8) | (loaded & 0xffu);
        tc::mbar_arrive_expect_tx(
            full, static_cast<uint32_t>(__popc(loaded)) *
                      static_cast<uint32_t>(which == 0 ? C::kHalvesK : C::kHalvesV) * C::kPieceBytes);
      }
      __syncwarp();
      if (MLA && my_piece && blk >= 0) {
        // Token row (request i, position tok0 + 16 pc) of the workspace.
        const int row = static_cast<int>(static_cast<long long>(i) * a.mla_s_max + tok0 + 16 * pc);
        const int halves = which == 0 ? C::kHalvesK : C::kHalvesV;
        for (int h = 0; h < halves; ++h)
          tc::tma_load_3d(dst + h * (C::kBN * 128) + pc * C::kPieceBytes,
                          which == 0 ? &kv_map : &v_map, full, h * 64, kvh, row);
      } else if (!MLA && my_piece && blk >= 0 && which == 1) {
        // V: both halves of the piece in one box (tensor map coordinates:
        // column 0, token, half 0, head, 2 * block + 1).
        tc::tma_load_5d(dst + pc * kVPiece, &v_map, full, 0, (tok0 + 16 * pc) % bs, 0, kvh,
                        2 * blk + 1);
      } else if (!MLA && my_piece && blk >= 0) {
#pragma unroll
        for (int h = 0; h < C::kHalvesK; ++h) {
          tc::tma_load_5d(dst + h * (C::kBN * 128) + pc * C::kPieceBytes, &kv_map, full, h * 64, kvh,
                          (tok0 + 16 * pc) % bs, which, blk);
        }
      }
    };
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    };
#ifdef PA_TEST_HOOKS
    const long long cta_id = blockIdx.x + static_cast<long long>(gridDim.x) *
                                              (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
    auto skipped = [&](int j) { return cta_id == g_test_skip.x && j == g_test_skip.y; };
#else
    auto skipped = [](int) { return false; };
#endif
    // K(j) and V(j) go to stage j & 1; stage reuse waits for S(j-2) / PV(j-2).
    auto issue_k = [&](int j, int blk) -> bool {
      const int st = j & 1;
      if (j >= 2 && !wait_all(BAR(kKEmpty + st), ((j >> 1) - 1) & 1)) return false;
      if (!skipped(j)) issue(j, blk, 0, sbase + C::kOffK + st * C::kKBytes, BAR(kKFull + st));
      return true;
    };
    auto issue_v = [&](int j, int blk) -> bool {
      const int vst = j % C::kVStages;
      if (j >= C::kVStages && !wait_all(BAR(kVEmpty + vst), ((j / C::kVStages) - 1) & 1))
        return false;
      if (!skipped(j)) issue(j, blk, 1, sbase + C::kOffV + vst * C::kVBytes, BAR(kVFull + vst));
      return true;
    };
    int r0 = raw_of(0), r1 = raw_of(1), r2 = raw_of(2);   // tiles j, j+1, j+2 (raw)
    tc::cluster_wait();
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    if (ntiles > 0) { ok = issue_k(0, valid_of(0, r0)); k_issued = 1; }
    if (ok && ntiles > 1) { ok = issue_k(1, valid_of(1, r1)); k_issued = 2; }
    for (int j = 0; ok && j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      if (!issue_v(j, valid_of(j, r0))) { ok = false; break; }
      v_issued = j + 1;
      const int r3 = raw_of(j + 3);   // in flight while K(j+2) waits for its stage
      if (j + 2 < ntiles) {
        if (!issue_k(j + 2, valid_of(j + 2, r2))) { ok = false; break; }
        k_issued = j + 3;
      }
      r0 = r1;
      r1 = r2;
      r2 = r3;
    }
    if (lane == 0) {
      if (!ok) fail();
      // No copy may still be landing when the CTA exits.
      for (int j = max(0, k_issued - 2); j < k_issued; ++j)
        if (!tc::mbar_wait(BAR(kKFull + (j & 1)), (j >> 1) & 1)) fail();
      for (int j = max(0, v_issued - C::kVStages); j < v_issued; ++j)
        if (!tc::mbar_wait(BAR(kVFull + j % C::kVStages), (j / C::kVStages) & 1)) fail();
    }
  } else {
    tc::cluster_wait();   // idle warps
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base(), C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

namespace {

// 5-D view of the standard pool [nb][2][bs][Hkv][d] (innermost first) with a
// 64-element x 1 head x 16 token box and 128-byte swizzle.
bool make_kv_map(CUtensorMap* map, const void* cache, int nb, int bs, int Hkv, int d) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Hkv),
                              static_cast<cuuint64_t>(bs), 2, static_cast<cuuint64_t>(nb)};
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2;
  const cuuint64_t strides[4] = {row, row * Hkv, row * Hkv * bs, row * Hkv * bs * 2};
  const cuuint32_t box[5] = {64, 1, 16, 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The V half of the same pool viewed 5-D so that one box holds a 16-token
// piece's 64-column halves as consecutive 128-byte-swizzled [16][128 B]
// tiles: dims (innermost first) 64 columns, bs tokens, d/64 halves, Hkv
// heads, 2 nb (kv index + 2 * block); box 64 x 16 x d/64 x 1 x 1.
bool make_v_map(CUtensorMap* map, const void* cache, int nb, int bs, int Hkv, int d) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(d / 64),
                              static_cast<cuuint64_t>(Hkv), 2 * static_cast<cuuint64_t>(nb)};
  const cuuint64_t row = static_cast<cuuint64_t>(d) * 2;
  const cuuint64_t strides[4] = {row * Hkv, 128, row, row * Hkv * bs};
  const cuuint32_t box[5] = {64, 16, static_cast<cuuint32_t>(d / 64), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// MLA prefill workspaces [rows][H][width] viewed 3-D (innermost first):
// 64-column x 1-head x 16-token boxes, 128-byte swizzle.
bool make_ws_map(CUtensorMap* map, const void* ws, long long rows, int H, int width) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(width) * 2,
                                 static_cast<cuuint64_t>(width) * 2 * H};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ws), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DK, int DV, int BN, int VST, bool EXT, bool MLA>
static cudaError_t launch_varlen_tc_t(const VarlenLaunch& L, cudaStream_t stream) {
  using C = TcCfg<DK, DV, BN, VST>;
  CUtensorMap map, vmap;
  if (MLA) {
    const long long rows = static_cast<long long>(L.N) * L.mla_s_max;
    if (!make_ws_map(&map, L.mla_k, rows, L.Hkv, DK) || !make_ws_map(&vmap, L.mla_v, rows, L.Hkv, DV))
      return cudaErrorInvalidValue;
  } else {
    // TMA coordinates are 32-bit: 2 * block + 1 must fit.
    if (2LL * L.num_blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (!make_kv_map(&map, L.cache, L.num_blocks, L.bs, L.Hkv, DK) ||
        !make_v_map(&vmap, L.cache, L.num_blocks, L.bs, L.Hkv, DV))
      return cudaErrorInvalidValue;
  }
  auto kern = varlen_tc_kernel<DK, DV, BN, VST, EXT, MLA>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  // The register hand-over between warpgroups waits for registers that the
  // launch must actually hold; refuse to launch a build that does not.
  static const bool regs_ok = [&] {
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return false;
    const long long have = static_cast<long long>(fa.numRegs) * C::kThreads;
    const long long need = 256LL * C::kRegSoftmax + 128LL * C::kRegOther;
    return fa.numRegs >= static_cast<int>(C::kRegOther) &&
           fa.numRegs <= static_cast<int>(C::kRegSoftmax) && have >= need;
  }();
  if (!regs_ok) return cudaErrorInvalidConfiguration;
  const bool virt = L.virt_total_q > 0;
  const long long qrows = virt ? L.virt_total_q : L.max_query_len;
  const long long rows = qrows * (L.Hq / L.Hkv);
  long long tiles = (rows + C::kRows - 1) / C::kRows;
  const int splits = L.kv_splits > 1 ? L.kv_splits : 1;
  if (tiles * splits > 0x7fffffffLL) return cudaErrorInvalidValue;
  VarlenArgs a{};
  a.q = static_cast<const __nv_bfloat16*>(L.q);
  a.block_table = L.block_table;
  a.qsl = L.qsl;
  a.seq_lens = L.seq_lens;
  a.max_blocks = L.max_blocks;
  a.Hq = L.Hq;
  a.Hkv = L.Hkv;
  a.bs = L.bs;
  a.num_blocks = L.num_blocks;
  a.scale_log2 = L.scale * kLog2e;
  a.causal = L.causal;
  a.window = L.window;
  a.out = static_cast<__nv_bfloat16*>(L.out);
  a.lse = L.lse;
  a.err = L.err;
  a.table_col0 = L.table_col0;
  a.seq_off = L.seq_off;
  a.virt_total_q = L.virt_total_q;
  a.virt_seq = L.virt_seq;
  a.ws = L.ws;
  a.ws_slots = L.ws_slots;
  a.ws_slot0 = L.ws_slot0;
  a.kv_splits = splits;
  a.kv_chunk = L.kv_chunk;
  a.mla_s_max = L.mla_s_max;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * splits), L.Hkv, virt ? 1 : L.N);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  // A cluster of one CTA (the kernel's start-up uses the cluster barrier).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, vmap, a);
}

#ifdef PA_TEST_HOOKS
// Test builds only (not declared in pa.h): makes the producer of CTA `cta`
// (linear block index) of the following varlen launches skip K/V tile `tile`;
// cta < 0 turns it off.
extern "C" int pa_test_skip_tile_loads(int cta, int tile) {
  const int2 v = make_int2(cta, tile);
  return cudaMemcpyToSymbol(g_test_skip, &v, sizeof(v)) == cudaSuccess ? 0 : 3;
}
#endif

cudaError_t launch_varlen_tc(const VarlenLaunch& L, cudaStream_t stream) {
  if (L.mla_k != nullptr)   // MLA prefill attention: [nope | rope] keys, 128-wide values
    return launch_varlen_tc_t<192, 128, 128, 1, false, true>(L, stream);
  const bool ext = L.window > 0 || L.kv_splits > 1 || L.ws != nullptr || L.virt_total_q > 0 ||
                   L.table_col0 != 0 || L.seq_off != 0;
  if (L.d == 128)
    return ext ? launch_varlen_tc_t<128, 128, 128, 2, true, false>(L, stream)
               : launch_varlen_tc_t<128, 128, 128, 2, false, false>(L, stream);
  return ext ? launch_varlen_tc_t<64, 64, 128, 2, true, false>(L, stream)
             : launch_varlen_tc_t<64, 64, 128, 2, false, false>(L, stream);
}

}  // namespace pa
