// MLA latent decode on tcgen05 tensor cores ("Triton and MLA" (vllm-arch-zh),
// data-flow section: MQA over one latent KV head).  The cache row of a token
// is the 576-wide [kv_c (512) | k_pe (64)] vector: the key is the whole row,
// the value its first 512 entries, so every cache byte is read from HBM once
// and serves both products.  Split-KV stage 1: each split writes its
// normalised partial output and LSE to the [B, H, S, 513] fp32 workspace;
// the LSE merge finishes the call.
//
// One (split, request, group of 128 heads) is computed by a cluster of two
// CTAs.  The 128 heads form the M = 128 rows of every MMA.  A 128 x 576 query
// (144 KB) and a 128 x 512 fp32 output (all 512 TMEM columns) do not fit one
// CTA next to a K ring and the scores, so the pair splits both:
//   * the contraction: CTA r holds the query / key columns of latent chunks
//     [256r, 256r + 256) and rope half [512 + 32r, 512 + 32r + 32); it computes
//     the partial scores S_r(j) = Q_r K_r(j)^T of a 64-token tile (N = 64);
//   * the output: CTA r accumulates O[:, 256r : 256r + 256], whose values are
//     exactly the latent columns it already holds.
// The partial scores are exchanged through distributed shared memory
// (st.async into the peer's buffer, completing bytes on the peer's barrier)
// as 16-bit fixed point: the SM-to-SM path moves only ~12 bytes per clock,
// and halving the bytes keeps the exchange behind the tensor core.  Each
// head row of a tile travels in units of a = max |S_peer| / 32767 over the
// row's visible tokens (the unit itself is sent with the row), rounded to
// int16, so the error of a score is at most a / 2 = max |S_peer| / 65534
// (f16 would allow 2^-12 of each value, ~16x more for the largest scores,
// which dominate the LSE; a power-of-two unit would waste up to one bit).
// CTA r then holds
// S = S_r + decode(S_peer) and runs the online softmax on it; each CTA's
// output half and row sum come from its own P, so each half is normalised
// consistently.  The query's latent half is the A operand of the score MMAs
// straight from TMEM (so shared memory holds only its 8 KB rope part and a
// four-stage K ring), and P goes to a shared-memory buffer that PV reads as
// its A operand, so the next scores can be computed into the S buffer as
// soon as the S of the tile has been read.
//
// 352 threads per CTA:
//   warps 0-3  softmax: thread t owns head t = TMEM lane t;
//   warps 4-7  exchange: as soon as S_r(j) has landed, thread t sends row t
//              of it to the peer, while the softmax warps still work on tile
//              j - 1 (the scores are double-buffered, so S_r(j) is computed
//              during the softmax of j - 1);
//   warp 8     MMA issue (one thread): S(j+2) as soon as S(j) has been read
//              (and K(j+2) has landed), PV(j) as soon as P(j) is written,
//              whichever comes first, so the scores of the next tiles are
//              computed while the softmax works on the current one;
//   warp 9     TMA producer: the query's rope half once, then per 64-token tile
//              two 32-token halves (each inside one cache block, since
//              block_size % 32 == 0) of 4 latent boxes (64 columns) and one
//              rope box (32 columns), through the block table;
//   warp 10    exchange helper: once the softmax warps have read the peer's
//              partial scores of a tile, tells the peer its buffer is free
//              (a thread with no remote stores of its own in flight, so the
//              cluster-scope release does not wait for them).  The query's
//              latent half is staged through the exchange buffers, so the
//              first "buffer free" of each buffer comes from the softmax
//              warps once they have read the query back.
// O is rescaled only when a head's running max grows by more than 2^8
// (exact: P keeps the older reference max).
//
// Shared memory per CTA (1024-byte aligned regions):
//   Qr    rope half of the query [128 heads][64 B] (64-byte swizzle)    8 KB
//   K/V   4 stages x (4 latent chunks [64 tokens][128 B] + rope half
//         [64 tokens][64 B])                                          144 KB
//   X     2 buffers of the peer's partial scores, [9 chunks][128 heads]
//         [16 B]: 8 chunks of 8 int16 scores, then the row's unit a, so
//         that one warp-wide store or load covers 512 contiguous bytes 36 KB
//   P     2 buffers [128 heads][64 tokens] bf16 (128-byte swizzle)     32 KB
// TMEM: S buffers at columns 0 and 64, the query's latent half (bf16 pairs)
// at 128-255, O half at columns 256-511.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"
#include "tc_common.cuh"

namespace pa {

struct MlaTcCfg {
  static constexpr int kDk = 576, kDv = 512, kH = 128, kBN = 64, kBox = 32;
  static constexpr int kLat = 4;                           // latent chunks per CTA
  static constexpr int kQRopeBytes = kH * 64;              // 8 KB
  static constexpr int kKChunkBytes = kBN * 128;           // 8 KB
  static constexpr int kKRopeBytes = kBN * 64;             // 4 KB
  static constexpr int kStageBytes = kLat * kKChunkBytes + kKRopeBytes;   // 36 KB
  static constexpr int kStages = 4;
  static constexpr int kHalfBytes = kBox * (kLat * 128 + 64);           // 18 KB per 32 tokens
  static constexpr int kXBytes = kH * 9 * 16;              // 18 KB per buffer
  static constexpr int kOffQr = 0;
  static constexpr int kOffK = kQRopeBytes;                // 8 KB
  static constexpr int kPBytes = kH * 128;                 // P tile: [128 heads][64 tokens] bf16
  static constexpr int kOffX = kOffK + kStages * kStageBytes;   // 152 KB
  static constexpr int kOffP = kOffX + 2 * kXBytes;        // 188 KB
  static constexpr int kOffBar = kOffP + 2 * kPBytes;      // 220 KB
  static constexpr int kBarBlock = 320;                    // barriers, TMEM slot, flags, ring
  static constexpr int kSmemBytes = kOffBar + kBarBlock + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColQ = 128;                   // query latent half, bf16 pairs
  static constexpr uint32_t kColO = 256;
  static constexpr int kThreads = 352;
};

enum MlaBar {
  kMQFull = 0,
  kMKFull = 1,                              // [kStages]
  kMKEmpty = kMKFull + MlaTcCfg::kStages,   // [kStages]
  kMSFull = kMKEmpty + MlaTcCfg::kStages,   // [2]
  kMXFull = kMSFull + 2,    // [2] the peer's partial scores have arrived in buffer b
  kMXEmpty = kMXFull + 2,   // [2] the peer has consumed buffer b of the scores this CTA sent
  kMPFull = kMXEmpty + 2,   // [2] P buffer b written
  kMPDone = kMPFull + 2,    // [2] PV of P buffer b completed
  kMFinal = kMPDone + 2,
  kMXRead = kMFinal + 1,    // [2] the softmax warps have read exchange buffer b
  kMSRead = kMXRead + 2,    // [2] the softmax and exchange warps have read S buffer b
  kMNumBars = kMSRead + 2
};
// Block layout after the barriers: TMEM slot (+0), abort flag (+8),
// descriptor ring (+16, kMlaRing words), rank pick (+16 + 4 * kMlaRing).
static_assert(8 * kMNumBars + 16 + 4 * 8 + 4 <= MlaTcCfg::kBarBlock,
              "MLA barrier block overflows its reservation");
// Tile descriptors passed from the producer: it runs up to kStages tiles
// ahead of the consumers, so the ring must hold more entries than that.
constexpr int kMlaRing = 8;
static_assert(kMlaRing > MlaTcCfg::kStages, "descriptor ring shorter than the producer's lead");
constexpr int kMlaRankMax = 512;    // largest batch ranked by seq_len (B^2 comparisons)

__device__ __forceinline__ uint32_t msw128(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ float mex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// x += a0 * b, y += a1 * b as one packed fp32 pair FMA.
__device__ __forceinline__ void ffma2_acc(float& x, float& y, float a0, float a1, float b) {
  asm("{\n.reg .b64 a, b, c;\nmov.b64 a, {%2, %3};\nmov.b64 b, {%4, %4};\n"
      "mov.b64 c, {%0, %1};\nfma.rn.f32x2 c, a, b, c;\nmov.b64 {%0, %1}, c;\n}"
      : "+f"(x), "+f"(y)
      : "f"(a0), "f"(a1), "f"(b));
}

__device__ __forceinline__ float mmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// Byte offset of 16-byte chunk c (0-8) of head row t in an exchange buffer.
__device__ __forceinline__ uint32_t xoff(int t, int c) {
  return static_cast<uint32_t>(c * 2048 + t * 16);
}

// The exchange's 16-bit fixed point, offset binary: a partial score x of a
// row with max |x| = amax travels as u = q + 32768, q = x * (32767 / amax)
// rounded to the nearest integer (nearest even; +32768 clamped to 32767),
// two per 32-bit word; the receiver scales q by a = amax / 32767.
// Integer <-> float conversions go through a bias, which keeps the exchange
// on the FMA and integer pipes: x * mul + (1.5 * 2^23 + 32768), rounded once
// by the FMA, is the float 1.5 * 2^23 + u, whose bits are 0x4B40 << 16 | u
// for 0 <= u < 2^16.  One byte permute packs a pair's low halves; the
// receiver rebuilds each float with one byte permute, subtracts the bias
// (exact: both are integers below 2^24) and adds q * a to its own partial
// score with one FMA.
constexpr float kXBias = 12615680.0f;   // 1.5 * 2^23 + 32768
constexpr uint32_t kXBiasHi = 0x4B40u;  // upper 16 bits of the float 1.5 * 2^23 + u
__device__ __forceinline__ uint32_t pack_q16(float lo, float hi, float mul) {
  float a, b;
  ffma2(a, b, lo, hi, mul, kXBias);
  a = fminf(a, kXBias + 32767.f);
  b = fminf(b, kXBias + 32767.f);
  return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x5410);
}

__global__ void __launch_bounds__(352, 1)
mla_tc_kernel(const __nv_bfloat16* __restrict__ q, const __grid_constant__ CUtensorMap qr_map,
              const __grid_constant__ CUtensorMap c_map, const __grid_constant__ CUtensorMap cr_map,
              const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
              int max_blocks, int H, int bs, int num_blocks, float scale_log2, int S, int chunk,
              float* __restrict__ ws, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
              int direct, int* err) {
  using C = MlaTcCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);

  const uint32_t rank = tc::cluster_rank();           // 0 or 1
  const uint32_t peer = rank ^ 1u;
  const int s = blockIdx.x >> 1, hg = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Pair row y of the grid takes the request of rank y in decreasing
  // seq_len (ties by index), so that the longest requests are dispatched
  // first and the last wave holds the short ones.  Every CTA ranks the whole
  // batch itself (B^2 / 352 comparisons, in the exchange buffers, which are
  // unused until after the cluster barrier below); batches above
  // kMlaRankMax keep the grid order.
  int b = blockIdx.y;
  if (gridDim.y <= kMlaRankMax) {
    // The lengths are padded with -1 (below every length) to a multiple of
    // four, so that each thread reads them as 16-byte vectors.
    const int nb = static_cast<int>(gridDim.y), nb4 = (nb + 3) >> 2;
    int* sl = reinterpret_cast<int*>(sgen + C::kOffX);
    volatile int* pick =
        reinterpret_cast<volatile int*>(sgen + C::kOffBar + 8 * kMNumBars + 16 + 4 * kMlaRing);
    for (int i = threadIdx.x; i < 4 * nb4; i += blockDim.x) sl[i] = i < nb ? seq_lens[i] : -1;
    __syncthreads();
    const int4* sl4 = reinterpret_cast<const int4*>(sl);
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
      const int v = sl[i];
      int rnk = 0;
#pragma unroll 8
      for (int k = 0; k < nb4; ++k) {
        const int4 u = sl4[k];
        rnk += (u.x > v || (u.x == v && 4 * k < i)) ? 1 : 0;
        rnk += (u.y > v || (u.y == v && 4 * k + 1 < i)) ? 1 : 0;
        rnk += (u.z > v || (u.z == v && 4 * k + 2 < i)) ? 1 : 0;
        rnk += (u.w > v || (u.w == v && 4 * k + 3 < i)) ? 1 : 0;
      }
      if (rnk == static_cast<int>(blockIdx.y)) *pick = i;
    }
    __syncthreads();
    b = *pick;
  }
  const int seq = seq_lens[b];
  const long long a0 = static_cast<long long>(s) * chunk;
  const int t0 = static_cast<int>(a0 < seq ? a0 : seq);
  const int t1 = (s == S - 1) ? seq : static_cast<int>(a0 + chunk < seq ? a0 + chunk : seq);
  const int ntiles = (t1 - t0 + C::kBN - 1) / C::kBN;
  const int32_t* table = block_table + static_cast<int64_t>(b) * max_blocks;

  const uint32_t bars = sbase + C::kOffBar;
  auto BAR = [&](int k) { return bars + 8u * static_cast<uint32_t>(k); };
  const uint32_t tmem_slot = bars + 8u * kMNumBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 8 * kMNumBars + 8);
  volatile uint32_t* ring =
      reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kMNumBars + 16);

  if (threadIdx.x == 0) {
    // The query: 128 softmax threads store its latent half in TMEM, the
    // producer's rope box lands by TMA.
    tc::mbar_init(BAR(kMQFull), 129);
    for (int k = 0; k < C::kStages; ++k) {
      tc::mbar_init(BAR(kMKFull + k), 1);
      tc::mbar_init(BAR(kMKEmpty + k), 1);
    }
    tc::mbar_init(BAR(kMSFull + 0), 1);
    tc::mbar_init(BAR(kMSFull + 1), 1);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(BAR(kMXFull + k), 1);
      tc::mbar_init(BAR(kMXEmpty + k), 1);   // the peer: its softmax warps, then its helper
      tc::mbar_init(BAR(kMXRead + k), 128);
    }
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(BAR(kMPFull + k), 128);
      tc::mbar_init(BAR(kMPDone + k), 1);
    }
    tc::mbar_init(BAR(kMFinal), 1);
    tc::mbar_init(BAR(kMSRead + 0), 256);
    tc::mbar_init(BAR(kMSRead + 1), 256);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_slot, C::kTmemCols);
  tc::tc_fence_before();
  // Both CTAs' barriers are initialised before either sends to the other.
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kMNumBars);

  auto fail = [&]() {
    record_error(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;   // head within the group
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t to = tmem + lane_base + C::kColO;
    const uint32_t xs = sbase + C::kOffX;
    auto all_ok = [&](bool w) -> bool {
      w = __all_sync(0xffffffffu, w);
      if (!w) fail();
      return w;
    };
    {
      // Head t's latent half of the query, [256 r, 256 r + 256), as the A
      // operand of the score MMAs: TMEM lane t, two bf16 per column (the
      // lower index in the low half).  The 512 bytes of each row come in
      // with one round of 16-byte asynchronous copies into the exchange and
      // P buffers (64 KB, unused until the first scores), chunk c of row t
      // at t * 512 + (c ^ (t & 7)) * 16 so that the reads back are free of
      // bank conflicts.
      const int head = hg * C::kH + t;
      const char* src = reinterpret_cast<const char*>(
          q + (static_cast<int64_t>(b) * H + (head < H ? head : 0)) * C::kDk + 256 * rank);
      const uint32_t stg = xs + static_cast<uint32_t>(t) * 512u;
#pragma unroll
      for (int c = 0; c < 32; ++c)
        cp_async_16(stg + ((c ^ (t & 7)) << 4), src + 16 * c, head < H ? 16 : 0);
      cp_async_commit();
      cp_async_wait<0>();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int v = 0; v < 8; ++v)
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(r[4 * v]), "=r"(r[4 * v + 1]), "=r"(r[4 * v + 2]), "=r"(r[4 * v + 3])
                       : "r"(stg + (((8 * c + v) ^ (t & 7)) << 4))
                       : "memory");
        tc::tmem_st32(tmem + lane_base + C::kColQ + c * 32, r);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kMQFull));
      // Once all 128 rows have been read back, the peer may send into the
      // exchange buffers: the first phase of both of its "buffer consumed"
      // barriers.
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (t == 0) {
        const uint32_t xempty_peer = tc::map_to_rank(BAR(kMXEmpty), peer);
        tc::mbar_arrive_remote(xempty_peer);
        tc::mbar_arrive_remote(xempty_peer + 8u);
      }
    }
    // l: the row's sum of weights (for the LSE); lr: the sum of the same
    // weights rounded to bf16, as PV multiplies them (for the output).
    float m_used = -CUDART_INF_F, l = 0.f, lr = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int buf = j & 1;
      const uint32_t ts = tmem + lane_base + 64u * buf;
      if (!all_ok(tc::mbar_wait(BAR(kMSFull + buf), (j >> 1) & 1))) break;
      tc::tc_fence_after();
      float sc[C::kBN];
      {
        uint32_t r[2][32];
        tc::tmem_ld32(ts, r[0]);
        tc::tmem_ld32(ts + 32, r[1]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          sc[e] = __uint_as_float(r[0][e]);
          sc[32 + e] = __uint_as_float(r[1][e]);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kMSRead + buf));
      // Add the peer's partial scores (sent by its exchange warps).
      if (t == 0) tc::mbar_arrive_expect_tx(BAR(kMXFull + buf), C::kXBytes);
      if (!all_ok(tc::mbar_wait_cluster(BAR(kMXFull + buf), (j >> 1) & 1))) break;
      {
        const uint32_t xb = xs + buf * C::kXBytes;
        uint32_t unit_bits;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(unit_bits) : "r"(xb + xoff(t, 8)) : "memory");
        const float unit = __uint_as_float(unit_bits);   // a = amax / 32767
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t v[4];
          asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                       : "r"(xb + xoff(t, c))
                       : "memory");
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            // The pair's two values q = (1.5 * 2^23 + u) - bias (exact), then
            // this CTA's partial scores += q * a; both steps as packed pairs.
            float d0 = __uint_as_float(__byte_perm(v[e], kXBiasHi, 0x5410));
            float d1 = __uint_as_float(__byte_perm(v[e], kXBiasHi, 0x5432));
            fadd2(d0, d1, -kXBias, -kXBias);
            ffma2_acc(sc[8 * c + 2 * e], sc[8 * c + 2 * e + 1], d0, d1, unit);
          }
        }
      }
      tc::mbar_arrive(BAR(kMXRead + buf));
      // Loaded halves of this tile, from the producer's ring.
      uint32_t vm;
      {
        const uint32_t tag = static_cast<uint32_t>(j) << 8;
        uint32_t w = ring[j % kMlaRing];
        for (int n = 0; (w & ~0xffu) != tag && n < tc::kWaitPolls; ++n) w = ring[j % kMlaRing];
        if (!all_ok((w & ~0xffu) == tag)) break;
        vm = w & 0x3u;
      }
      const int tok0 = t0 + j * C::kBN;
      const int nvis = min(C::kBN, t1 - tok0);   // tokens of the tile inside the split
      if (nvis < C::kBN || vm != 0x3u) {
#pragma unroll
        for (int e = 0; e < C::kBN; ++e) {
          const bool vis = e < nvis && ((vm >> (e >> 5)) & 1u);
          sc[e] = vis ? sc[e] : -CUDART_INF_F;
        }
      }
      float mx;
      {
        float m8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = fmaxf(sc[k], sc[8 + k]);
#pragma unroll
        for (int e = 16; e < C::kBN; e += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = mmax3(m8[k], sc[e + k], sc[e + 8 + k]);
        mx = mmax3(mmax3(m8[0], m8[1], m8[2]), mmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        mx *= scale_log2;
      }
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;
      const float alpha = need ? mex2(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
      // Rescale O once PV(j-1) and PV(j-2) have completed (PV(j-3) has:
      // it was issued before S(j)).
      if (__any_sync(0xffffffffu, need) && j > 0) {
        if (j >= 2 && !all_ok(tc::mbar_wait(BAR(kMPDone + buf), ((j >> 1) - 1) & 1))) break;
        if (!all_ok(tc::mbar_wait(BAR(kMPDone + (buf ^ 1)), ((j - 1) >> 1) & 1))) break;
        tc::tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 256 / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(to + c * 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tc::tmem_st32(to + c * 32, r);
        }
      }
      // Value rows that must contribute nothing (past the split, or in a half
      // that was not loaded) are zeroed: they may hold anything.
      if (t < C::kBN && !(t < nvis && ((vm >> (t >> 5)) & 1u))) {
        const uint32_t vb = sbase + C::kOffK + (j % C::kStages) * C::kStageBytes;
#pragma unroll
        for (int ch = 0; ch < C::kLat; ++ch)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vb + ch * C::kKChunkBytes +
                                                                     msw128(t, c)),
                         "r"(0u)
                         : "memory");
        tc::fence_proxy_async_smem();
      }
      // P = exp2(s * scale_log2 - m_used) as bf16, row t of shared-memory
      // P buffer `buf` (128-byte swizzle, the A operand of PV), once PV(j-2)
      // has read it.  Keeping P out of TMEM lets S(j+2) reuse the S buffer
      // as soon as S(j) has been read.  Two row sums: of the weights (the
      // LSE), and of the bf16-rounded weights that PV multiplies (the
      // output's divisor), so that the output is a weighted mean whose
      // weights sum to 1: where one token dominates, its value comes out
      // unscaled by the up to 2^-9 rounding of its weight.
      if (j >= 2 && !all_ok(tc::mbar_wait(BAR(kMPDone + buf), ((j >> 1) - 1) & 1))) break;
      {
        const uint32_t pb = sbase + C::kOffP + buf * C::kPBytes;
        float l8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float r8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x0, x1;
            ffma2(x0, x1, sc[8 * c + 2 * e], sc[8 * c + 2 * e + 1], scale_log2, -mu);
            const float p0 = mex2(x0);
            const float p1 = mex2(x1);
            fadd2(l8[2 * e], l8[2 * e + 1], p0, p1);
            pk[e] = pack_bf16(p0, p1);
            add_bf16x2_f32(r8[2 * e], r8[2 * e + 1], pk[e]);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(pb + msw128(t, c)),
                       "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                       : "memory");
        }
        l = l * alpha + (((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7])));
        lr = lr * alpha + (((r8[0] + r8[1]) + (r8[2] + r8[3])) + ((r8[4] + r8[5]) + (r8[6] + r8[7])));
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(BAR(kMPFull + buf));
    }
    // ------------------------------------------------------------ epilogue
    bool ok = !__any_sync(0xffffffffu, *abort_flag != 0) && ntiles > 0;
    // Every MMA has completed once the final commit has landed.
    if (ok) ok = all_ok(tc::mbar_wait(BAR(kMFinal), 0));
    tc::tc_fence_after();
    const int head = hg * C::kH + t;
    // One split: the output row (bf16) and LSE directly; else the split's
    // partial row of the workspace.
    float* dst = ws + ((static_cast<int64_t>(b) * H + head) * S + s) * (C::kDv + 1);
    uint4* orow = reinterpret_cast<uint4*>(out + (static_cast<int64_t>(b) * H + head) * C::kDv +
                                           256 * rank);
    const float lse_v = (ok && l > 0.f) ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
    if (ok) {   // warp-uniform: TMEM loads are collective
      const float inv = lr > 0.f ? 1.f / lr : 0.f;
#pragma unroll 1
      for (int c = 0; c < 256 / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(to + c * 32, r);
        tc::tmem_wait_ld();
        if (head < H && direct) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(r[v * 8 + 0]) * inv, __uint_as_float(r[v * 8 + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(r[v * 8 + 2]) * inv, __uint_as_float(r[v * 8 + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(r[v * 8 + 4]) * inv, __uint_as_float(r[v * 8 + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(r[v * 8 + 6]) * inv, __uint_as_float(r[v * 8 + 7]) * inv);
            orow[c * 4 + v] = w;
          }
        } else if (head < H) {
#pragma unroll
          for (int e = 0; e < 32; ++e) dst[256 * rank + c * 32 + e] = __uint_as_float(r[e]) * inv;
        }
      }
    } else if (head < H) {
      // Nothing visible (or an aborted pair): o = 0, lse = -inf.
      if (direct)
        for (int e = 0; e < 32; ++e) orow[e] = make_uint4(0, 0, 0, 0);
      else
        for (int e = 0; e < 256; ++e) dst[256 * rank + e] = 0.f;
    }
    if (head < H && rank == 0) {
      if (!direct)
        dst[C::kDv] = lse_v;
      else if (lse != nullptr)
        lse[static_cast<int64_t>(b) * H + head] = lse_v;
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ exchange
    const int t = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t x_peer = tc::map_to_rank(sbase + C::kOffX, peer);
    const uint32_t xfull_peer = tc::map_to_rank(BAR(kMXFull), peer);
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int buf = j & 1;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(BAR(kMSFull + buf), (j >> 1) & 1))) {
        fail();
        break;
      }
      tc::tc_fence_after();
      uint32_t r[2][32];
      tc::tmem_ld32(tmem + lane_base + 64u * buf, r[0]);
      tc::tmem_ld32(tmem + lane_base + 64u * buf + 32, r[1]);
      tc::tmem_wait_ld();
      // Visible tokens of the tile (descriptor from the producer's ring, read
      // before S buffer `buf` is released): the others may hold anything and
      // are sent as 0.
      uint32_t vm;
      {
        const uint32_t tag = static_cast<uint32_t>(j) << 8;
        uint32_t w = ring[j % kMlaRing];
        for (int n = 0; (w & ~0xffu) != tag && n < tc::kWaitPolls; ++n) w = ring[j % kMlaRing];
        if (!__all_sync(0xffffffffu, (w & ~0xffu) == tag)) {
          fail();
          break;
        }
        vm = w & 0x3u;
      }
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kMSRead + buf));
      const int nvis = min(C::kBN, t1 - (t0 + j * C::kBN));
      float v[C::kBN];
#pragma unroll
      for (int e = 0; e < C::kBN; ++e) v[e] = __uint_as_float(r[e >> 5][e & 31]);
      if (nvis < C::kBN || vm != 0x3u) {
#pragma unroll
        for (int e = 0; e < C::kBN; ++e) {
          const bool vis = e < nvis && ((vm >> (e >> 5)) & 1u);
          v[e] = vis ? v[e] : 0.f;
        }
      }
      float a8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) a8[k] = fmaxf(fabsf(v[k]), fabsf(v[8 + k]));
#pragma unroll
      for (int e = 16; e < C::kBN; e += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) a8[k] = mmax3(a8[k], fabsf(v[e + k]), fabsf(v[e + 8 + k]));
      const float amax = mmax3(mmax3(a8[0], a8[1], a8[2]), mmax3(a8[3], a8[4], a8[5]),
                               fmaxf(a8[6], a8[7]));
      // The row's unit a = amax / 32767 and its inverse (0 for an all-zero
      // row, whose codes are then all 0).
      const float unit = amax * (1.f / 32767.f);
      const float mul = amax > 0.f ? 32767.f * __frcp_rn(amax) : 0.f;
      // The peer has consumed what this CTA sent into buffer `buf` two
      // tiles ago.
      if (!__all_sync(0xffffffffu, tc::mbar_wait_cluster(BAR(kMXEmpty + buf), (j >> 1) & 1))) {
        fail();
        break;
      }
      const uint32_t dst = x_peer + buf * C::kXBytes;
      const uint32_t full = xfull_peer + 8u * buf;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int e = c * 8;
        tc::st_async_v4(dst + xoff(t, c), pack_q16(v[e], v[e + 1], mul),
                        pack_q16(v[e + 2], v[e + 3], mul), pack_q16(v[e + 4], v[e + 5], mul),
                        pack_q16(v[e + 6], v[e + 7], mul), full);
      }
      tc::st_async_v4(dst + xoff(t, 8), __float_as_uint(unit), 0u, 0u, 0u, full);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, C::kBN, 0, 0);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(128, 256, 0, 1);
      const uint32_t qr = sbase + C::kOffQr;
      // S(j) = Q_r K_r(j)^T into S buffer j & 1: the latent half with A from
      // TMEM (16 K-steps of 8 columns) against the 4 latent chunks of the
      // stage (128-byte swizzle), then the rope half from shared memory
      // (2 K-steps, 64-byte swizzle).
      auto issue_s = [&](int j) {
        const uint32_t ks = sbase + C::kOffK + (j % C::kStages) * C::kStageBytes;
        const uint32_t d = tmem + 64u * (j & 1);
#pragma unroll
        for (int c = 0; c < C::kLat; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ts(d, tmem + C::kColQ + (c * 4 + kk) * 8,
                            tc::smem_desc_sw128(ks + c * C::kKChunkBytes + kk * 32, 16, 1024),
                            idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          tc::mma_bf16_ss(d, tc::smem_desc_sw64(qr + kk * 32, 512),
                          tc::smem_desc_sw64(ks + C::kLat * C::kKChunkBytes + kk * 32, 512),
                          idesc_s, 1u);
        tc::mma_commit(BAR(kMSFull + (j & 1)));
      };
      auto wait_k = [&](int j) {
        return tc::mbar_wait(BAR(kMKFull + j % C::kStages), (j / C::kStages) & 1);
      };
      // O_r += P(j) V_r(j): P from shared-memory buffer j & 1 (K-major,
      // 32 bytes = 16 tokens per K-step), V_r = the 4 latent chunks of the
      // stage, N = 256.
      auto issue_pv = [&](int j) {
        const uint32_t vs = sbase + C::kOffK + (j % C::kStages) * C::kStageBytes;
        const uint32_t pa = sbase + C::kOffP + (j & 1) * C::kPBytes;
#pragma unroll
        for (int k = 0; k < C::kBN / 16; ++k)
          tc::mma_bf16_ss(tmem + C::kColO, tc::smem_desc_sw128(pa + k * 32, 16, 1024),
                          tc::smem_desc_sw128(vs + k * 16 * 128, C::kKChunkBytes, 1024), idesc_o,
                          (j > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(BAR(kMPDone + (j & 1)));
        tc::mma_commit(BAR(kMKEmpty + j % C::kStages));
      };
      bool ok = ntiles == 0 || tc::mbar_wait(BAR(kMQFull), 0);
      for (int j = 0; ok && j < 2 && j < ntiles; ++j) {
        ok = wait_k(j);
        if (ok) {
          tc::tc_fence_after();
          issue_s(j);
        }
      }
      // Per tile j: PV(j) once P(j) is written, and S(j+2) into S buffer
      // j & 1 once S(j) has been read from it and K(j+2) has landed, in
      // whichever order they become ready -- PV first when both are, since
      // the tensor pipe runs in issue order and PV(j) frees the K stage that
      // a later K load is waiting for.
      for (int j = 0; ok && j < ntiles; ++j) {
        bool s_done = j + 2 >= ntiles, pv_done = false;
        int n = 0;
        for (; n < tc::kWaitPolls && !(s_done && pv_done); ++n) {
          if (*abort_flag) break;
          if (!pv_done && tc::mbar_try_wait(BAR(kMPFull + (j & 1)), (j >> 1) & 1)) {
            tc::tc_fence_after();
            issue_pv(j);
            pv_done = true;
          }
          if (!s_done && tc::mbar_try_wait(BAR(kMSRead + (j & 1)), (j >> 1) & 1) &&
              tc::mbar_try_wait(BAR(kMKFull + (j + 2) % C::kStages), ((j + 2) / C::kStages) & 1)) {
            tc::tc_fence_after();
            issue_s(j + 2);
            s_done = true;
          }
        }
        if (!(s_done && pv_done)) ok = false;
      }
      if (!ok && !*abort_flag) fail();
      tc::mma_commit(BAR(kMFinal));
      if (!tc::mbar_wait(BAR(kMFinal), 0)) fail();
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    // Lane i < 10 owns box i % 5 (latent chunk 0-3, or the rope half) of the
    // 32-token half i / 5 of every tile.
    if (lane == 0) {
      tc::tma_prefetch_desc(&qr_map);
      tc::tma_prefetch_desc(&c_map);
      tc::tma_prefetch_desc(&cr_map);
    }
    const int half = lane / 5, box = lane % 5;
    const bool box_lane = lane < 10;
    if (ntiles > 0 && lane == 0) {
      tc::mbar_arrive_expect_tx(BAR(kMQFull), C::kQRopeBytes);
      tc::tma_load_2d_(sbase + C::kOffQr, &qr_map, BAR(kMQFull), 512 + 32 * static_cast<int>(rank),
                       b * H + hg * C::kH);
    }
    // Half `half` of tile j lies inside the split iff its first token does.
    auto in_split = [&](int j) -> bool {
      return box_lane && j < ntiles && t0 + j * C::kBN + half * C::kBox < t1;
    };
    // Raw table entry of that half (-1 outside the split or past the table).
    // Loaded three tiles ahead and validated only when used, so that the
    // load's latency never stalls the issue of the current tile.
    auto raw_block = [&](int j) -> int {
      if (!in_split(j)) return -1;
      const int idx = (t0 + j * C::kBN + half * C::kBox) / bs;
      return idx < max_blocks ? __ldg(table + idx) : -1;
    };
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    };
    int issued = 0;
    bool ok = true;
    // Raw ids of tiles j .. j+3 in rr[j % 4]: the loop is unrolled four
    // times so that every index is a constant and a load's value is first
    // touched three iterations after it was issued (a register rotation
    // would wait for it at once).
    int rr[4] = {raw_block(0), raw_block(1), raw_block(2), -1};
    bool go = true;
    for (int jb = 0; go && jb < ntiles; jb += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = jb + u;
        if (!go || j >= ntiles) continue;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          go = false;
          continue;
        }
        const int st = j % C::kStages;
        if (j >= C::kStages && !wait_all(BAR(kMKEmpty + st), ((j / C::kStages) - 1) & 1)) {
          ok = false;
          go = false;
          continue;
        }
        rr[(u + 3) & 3] = raw_block(j + 3);
        const int r0 = rr[u];
        // The id, -1 (outside the split) or -2 (invalid id).
        const int blk = !in_split(j) ? -1 : (r0 >= 0 && r0 < num_blocks) ? r0 : -2;
        // Lanes 0 and 5 speak for halves 0 and 1.
        const unsigned loaded = __ballot_sync(0xffffffffu, blk >= 0);
        const unsigned bad = __ballot_sync(0xffffffffu, blk == -2);
        const uint32_t mask = ((loaded >> 0) & 1u) | (((loaded >> 5) & 1u) << 1);
        const uint32_t full = BAR(kMKFull + st);
        if (lane == 0) {
          if (bad != 0u) record_error(err, PA_DEVERR_BLOCK_ID);
          ring[j % kMlaRing] = (static_cast<uint32_t>(j) << 8) | mask;
          tc::mbar_arrive_expect_tx(full, static_cast<uint32_t>(__popc(mask)) * C::kHalfBytes);
        }
        __syncwarp();
        if (blk >= 0) {
          const uint32_t stage = sbase + C::kOffK + st * C::kStageBytes;
          const int tok = (t0 + j * C::kBN + half * C::kBox) % bs;
          if (box < C::kLat)
            tc::tma_load_3d(stage + box * C::kKChunkBytes + half * (C::kBox * 128), &c_map, full,
                            256 * static_cast<int>(rank) + 64 * box, tok, blk);
          else
            tc::tma_load_3d(stage + C::kLat * C::kKChunkBytes + half * (C::kBox * 64), &cr_map,
                            full, 512 + 32 * static_cast<int>(rank), tok, blk);
        }
        issued = j + 1;
      }
    }
    if (lane == 0) {
      if (!ok) fail();
      // No copy may still be landing when the CTA exits.
      if (ntiles > 0 && !tc::mbar_wait(BAR(kMQFull), 0)) fail();
      for (int j = max(0, issued - C::kStages); j < issued; ++j)
        if (!tc::mbar_wait(BAR(kMKFull + j % C::kStages), (j / C::kStages) & 1)) fail();
    }
  } else if (warp == 10 && lane == 0) {
    // ------------------------------------------------------------ exchange helper
    const uint32_t xempty_peer = tc::map_to_rank(BAR(kMXEmpty), peer);
    for (int j = 0; j < ntiles; ++j) {
      bool w = false;
      for (int n = 0; n < tc::kWaitPolls && !w; ++n) {
        w = tc::mbar_try_wait(BAR(kMXRead + (j & 1)), (j >> 1) & 1);
        if (!w && *abort_flag) break;
      }
      if (!w) break;
      tc::mbar_arrive_remote(xempty_peer + 8u * (j & 1));
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
  // Neither CTA leaves while the other may still write into its shared
  // memory or arrive on its barriers.
  tc::cluster_sync();
}

// ---------------------------------------------------------------- host side

namespace {

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_mla_tc(const void* q, const void* cache, const int32_t* block_table,
                          const int32_t* seq_lens, int B, int H, int bs, int num_blocks,
                          int max_blocks, float scale, int S, int chunk, float* ws, void* out,
                          float* lse, int* err, cudaStream_t stream) {
  using C = MlaTcCfg;
  // Query [B*H rows][576]: 64-column latent boxes and 32-column rope boxes of
  // 128 heads.  Cache [nb][bs][576]: the same boxes over 32 tokens.
  CUtensorMap qr_map, c_map, cr_map;
  {
    const cuuint64_t dims[2] = {C::kDk, static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[1] = {C::kDk * 2};
    const cuuint32_t box_r[2] = {32, C::kH};
    if (!encode(&qr_map, q, 2, dims, strides, box_r, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {C::kDk, static_cast<cuuint64_t>(bs),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[2] = {C::kDk * 2, static_cast<cuuint64_t>(C::kDk) * 2 * bs};
    const cuuint32_t box[3] = {64, C::kBox, 1};
    const cuuint32_t box_r[3] = {32, C::kBox, 1};
    if (!encode(&c_map, cache, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode(&cr_map, cache, 3, dims, strides, box_r, CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
  }
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(mla_tc_kernel, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * S, B, (H + C::kH - 1) / C::kH);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // With one split each pair writes its output rows and LSE itself (16-byte
  // vector stores), and the workspace and the merge are skipped.
  const int direct = (S == 1 && (reinterpret_cast<uintptr_t>(out) & 15u) == 0) ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, mla_tc_kernel, static_cast<const __nv_bfloat16*>(q), qr_map, c_map,
                         cr_map, block_table, seq_lens,
                         max_blocks, H, bs, num_blocks, scale * kLog2e, S, chunk, ws,
                         static_cast<__nv_bfloat16*>(out), lse, direct, err);
  if (e != cudaSuccess || direct) return e;
  return launch_lse_merge(ws, B * H, S, C::kDv, out, lse, stream);
}

}  // namespace pa
