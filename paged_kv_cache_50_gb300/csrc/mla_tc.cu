// MLA latent decode on tcgen05 tensor cores ("Triton and MLA" (vllm-arch-zh),
// data-flow section: MQA over one latent KV head).  The cache row of a token
// is the 576-wide [kv_c (512) | k_pe (64)] vector: the key is the whole row,
// the value its first 512 entries, so every cache byte is read from HBM once
// and serves both products.  Split-KV stage 1: each CTA writes its split's
// normalised partial output and LSE to the [B, H, S, 513] fp32 workspace;
// the LSE merge finishes the call.
//
// CTA = (split, request, group of 128 heads); the 128 heads form the M = 128
// rows of every MMA (a last partial group computes spare rows it never stores).  192 threads:
//   warps 0-3  softmax: thread t owns head t = TMEM lane t;
//   warp 4     MMA issue (one thread);
//   warp 5     TMA producer: Q once (9 boxes of 64 columns x 128 heads), then
//              per 32-token tile 9 boxes of 64 columns x 32 tokens, one per
//              lane, from the token's cache block (block_size % 32 == 0).
// Tensor memory holds 512 fp32 columns per lane, exactly one 128 x 512 output,
// which leaves no room for the scores.  So O[:, 0:448] accumulates in TMEM
// columns 0-447, and columns 448-511 (region X) serve in turn as
//   S(j)    = Q K(j)^T             (32 columns), read by the softmax warps;
//   T(j)    = P(j) V(j)[:, 448:512] (64 columns), added by the softmax warps
//             into the last 64 output columns they keep in registers.
// Per tile: S(j) -> softmax -> P(j) -> PV(j) (O[:, 0:448] and T(j)) -> T(j)
// read back -> X free -> S(j+1).  O is rescaled only when a head's running
// max grows by more than 2^8 (exact: P keeps the older reference max).
//
// Shared memory: Q [9 chunks][128 heads][128 B] (144 KB, 128-byte swizzle),
// K/V tiles 2 stages x [9 chunks][32 tokens][128 B] (72 KB), P [128 heads]
// [32 tokens] bf16 in the unswizzled 8 x 16-byte core-matrix layout (8 KB).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_launch.h"
#include "tc_common.cuh"

namespace pa {

struct MlaTcCfg {
  static constexpr int kDk = 576, kDv = 512, kH = 128, kBN = 32;
  static constexpr int kChunks = kDk / 64;                 // 9 column chunks of 64
  static constexpr int kQChunkBytes = kH * 128;            // 16 KB
  static constexpr int kKChunkBytes = kBN * 128;           // 4 KB
  static constexpr int kStageBytes = kChunks * kKChunkBytes;  // 36 KB
  static constexpr int kPBytes = kH * kBN * 2;             // 8 KB
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kChunks * kQChunkBytes;     // 144 KB
  static constexpr int kOffP = kOffK + 2 * kStageBytes;    // 216 KB
  static constexpr int kOffBar = kOffP + kPBytes;          // 224 KB
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColX = 448;                   // S / tail region
  static constexpr int kMainCols = 448;
  static constexpr int kTailCols = kDv - kMainCols;        // 64
  static constexpr int kThreads = 192;
};

enum MlaBar { kMQFull = 0, kMKFull = 1, kMKEmpty = 3, kMSFull = 5, kMPFull = 6, kMPvDone = 7,
              kMXFree = 8, kMFinal = 9, kMNumBars = 10 };

__device__ __forceinline__ uint32_t msw128(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ float mex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory descriptor of an unswizzled K-major tile: 8-row x 16-byte
// core matrices, `lbo` bytes apart along K and `sbo` bytes apart along M/N.
__device__ __forceinline__ uint64_t smem_desc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

__global__ void __launch_bounds__(192, 1)
mla_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap c_map,
              const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
              int max_blocks, int H, int bs, int num_blocks, float scale_log2, int S, int chunk,
              float* __restrict__ ws, int* err) {
  using C = MlaTcCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  if (err != nullptr && (*reinterpret_cast<volatile int*>(err) & PA_DEVERR_TIMEOUT)) return;

  const int s = blockIdx.x, b = blockIdx.y, hg = blockIdx.z;   // hg: group of 128 heads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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

  if (threadIdx.x == 0) {
    tc::mbar_init(BAR(kMQFull), 1);
    for (int k = 0; k < 2; ++k) {
      tc::mbar_init(BAR(kMKFull + k), 1);
      tc::mbar_init(BAR(kMKEmpty + k), 1);
    }
    tc::mbar_init(BAR(kMSFull), 1);
    tc::mbar_init(BAR(kMPFull), 128);
    tc::mbar_init(BAR(kMPvDone), 1);
    tc::mbar_init(BAR(kMXFree), 128);
    tc::mbar_init(BAR(kMFinal), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) tc::tmem_alloc(tmem_slot, C::kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kMNumBars);

  auto fail = [&]() {
    record_error(err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  };
  // Block id of tile j (its 32 tokens lie in one cache block), or -1.
  auto tile_block = [&](int j) -> int {
    const int tok = t0 + j * C::kBN;
    const int blk = block_at(table, tok / bs, max_blocks);
    return (blk >= 0 && blk < num_blocks) ? blk : -1;
  };

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int t = threadIdx.x;   // head
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    auto wait_warp = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool w = __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
      if (!w) fail();
      return w;
    };
    float m_used = -CUDART_INF_F, l = 0.f;
    float tail[C::kTailCols];
#pragma unroll
    for (int e = 0; e < C::kTailCols; ++e) tail[e] = 0.f;
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int tok0 = t0 + j * C::kBN;
      const bool tile_ok = tile_block(j) >= 0;
      const int lim = tile_ok ? min(C::kBN, t1 - tok0) : 0;   // visible tokens of the tile
      if (!wait_warp(BAR(kMSFull), j & 1)) break;
      tc::tc_fence_after();
      float sc[C::kBN];
      {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lane_base + C::kColX, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < C::kBN; ++e) sc[e] = e < lim ? __uint_as_float(r[e]) : -CUDART_INF_F;
      }
      float mx;
      {
        float m4[4] = {sc[0], sc[1], sc[2], sc[3]};
#pragma unroll
        for (int e = 4; e < C::kBN; ++e) m4[e & 3] = fmaxf(m4[e & 3], sc[e]);
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * scale_log2;
      }
      const float m_new = fmaxf(m_used, mx);
      const bool need = m_new > m_used + 8.f;
      const float alpha = need ? mex2(m_used - m_new) : 1.f;
      if (need) m_used = m_new;
      const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
      uint32_t pk[C::kBN / 2];
      {
        float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < C::kBN / 2; ++c) {
          const float p0 = mex2(fmaf(sc[2 * c], scale_log2, -mu));
          const float p1 = mex2(fmaf(sc[2 * c + 1], scale_log2, -mu));
          l4[c & 3] += p0 + p1;
          pk[c] = pack_bf16(p0, p1);
        }
        l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
      }
      // PV(j-1) and its tail have completed (X was freed before S(j)), so O
      // can be rescaled here.
      if (__any_sync(0xffffffffu, need) && j > 0) {
#pragma unroll 1
        for (int c = 0; c < C::kMainCols / 32; ++c) {
          uint32_t r[32];
          const uint32_t ta = tmem + lane_base + c * 32;
          tc::tmem_ld32(ta, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
          tc::tmem_st32(ta, r);
        }
        tc::tmem_wait_st();
#pragma unroll
        for (int e = 0; e < C::kTailCols; ++e) tail[e] *= alpha;
      }
      // P row t: 32 tokens = 4 core-matrix columns of 16 bytes.
      {
        const uint32_t pbase = sbase + C::kOffP;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t dst = pbase + ((t >> 3) * 4 + c) * 128 + (t & 7) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(pk[4 * c]),
                       "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                       : "memory");
        }
      }
      // Value rows of tokens the tile must not contribute (past the split or
      // the whole tile when its block id is invalid) are zeroed: they may
      // hold anything.
      if (t < C::kBN && t >= lim) {
        const uint32_t vb = sbase + C::kOffK + (j & 1) * C::kStageBytes;
#pragma unroll
        for (int ch = 0; ch < C::kDv / 64; ++ch)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(vb + ch * C::kKChunkBytes +
                                                                     msw128(t, c)),
                         "r"(0u)
                         : "memory");
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kMPFull));
      // Tail T(j) = P(j) V(j)[:, 448:512] lands in X together with PV(j).
      if (!wait_warp(BAR(kMPvDone), j & 1)) break;
      tc::tc_fence_after();
      {
        uint32_t r[2][32];
        tc::tmem_ld32(tmem + lane_base + C::kColX, r[0]);
        tc::tmem_ld32(tmem + lane_base + C::kColX + 32, r[1]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          tail[e] += __uint_as_float(r[0][e]);
          tail[32 + e] += __uint_as_float(r[1][e]);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kMXFree));
    }
    // ------------------------------------------------------------ epilogue
    const bool ok = !__any_sync(0xffffffffu, *abort_flag != 0) && ntiles > 0;
    tc::tc_fence_after();
    const int head = hg * C::kH + t;
    float* dst = ws + ((static_cast<int64_t>(b) * H + head) * S + s) * (C::kDv + 1);
    if (head >= H) {
      // A row of the last, partial head group: computed, never stored.
    } else if (ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < C::kMainCols / 32; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lane_base + c * 32, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) dst[c * 32 + e] = __uint_as_float(r[e]) * inv;
      }
#pragma unroll
      for (int e = 0; e < C::kTailCols; ++e) dst[C::kMainCols + e] = tail[e] * inv;
      dst[C::kDv] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -CUDART_INF_F;
    } else {
      for (int e = 0; e < C::kDv; ++e) dst[e] = 0.f;
      dst[C::kDv] = -CUDART_INF_F;
    }
  } else if (warp == 4) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(128, C::kBN, 0, 0);
      constexpr uint32_t idesc_o256 = tc::idesc_bf16_f32(128, 256, 0, 1);
      constexpr uint32_t idesc_o192 = tc::idesc_bf16_f32(128, 192, 0, 1);
      constexpr uint32_t idesc_t64 = tc::idesc_bf16_f32(128, 64, 0, 1);
      const uint32_t qs = sbase + C::kOffQ, ps = sbase + C::kOffP;
      bool ok = ntiles == 0 || tc::mbar_wait(BAR(kMQFull), 0);
      for (int j = 0; ok && j < ntiles; ++j) {
        if (*abort_flag) { ok = false; break; }
        const int st = j & 1;
        if (!tc::mbar_wait(BAR(kMKFull + st), (j >> 1) & 1)) { ok = false; break; }
        if (j > 0 && !tc::mbar_wait(BAR(kMXFree), (j - 1) & 1)) { ok = false; break; }
        tc::tc_fence_after();
        const uint32_t ks = sbase + C::kOffK + st * C::kStageBytes;
        // S(j) = Q K(j)^T over the 576 columns: 9 chunks x 4 K-steps.
#pragma unroll 1
        for (int c = 0; c < C::kChunks; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ss(tmem + C::kColX,
                            tc::smem_desc_sw128(qs + c * C::kQChunkBytes + kk * 32, 16, 1024),
                            tc::smem_desc_sw128(ks + c * C::kKChunkBytes + kk * 32, 16, 1024),
                            idesc_s, (c > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit(BAR(kMSFull));
        if (!tc::mbar_wait(BAR(kMPFull), j & 1)) { ok = false; break; }
        tc::tc_fence_after();
        // O[:, 0:448] += P V[:, 0:448];  X = P V[:, 448:512].
#pragma unroll
        for (int k = 0; k < C::kBN / 16; ++k) {
          const uint64_t pd = smem_desc_noswz(ps + k * 2 * 128, 128, 512);
          const uint32_t vrow = ks + k * 16 * 128;
          const uint32_t acc = (j > 0 || k > 0) ? 1u : 0u;
          tc::mma_bf16_ss(tmem + 0, pd, tc::smem_desc_sw128(vrow, C::kKChunkBytes, 1024),
                          idesc_o256, acc);
          tc::mma_bf16_ss(tmem + 256, pd,
                          tc::smem_desc_sw128(vrow + 4 * C::kKChunkBytes, C::kKChunkBytes, 1024),
                          idesc_o192, acc);
          tc::mma_bf16_ss(tmem + C::kColX, pd,
                          tc::smem_desc_sw128(vrow + 7 * C::kKChunkBytes, C::kKChunkBytes, 1024),
                          idesc_t64, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(BAR(kMPvDone));
        tc::mma_commit(BAR(kMKEmpty + st));
      }
      if (!ok && !*abort_flag) fail();
      tc::mma_commit(BAR(kMFinal));
      if (!tc::mbar_wait(BAR(kMFinal), 0)) fail();
    }
  } else {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&q_map);
      tc::tma_prefetch_desc(&c_map);
    }
    auto wait_all = [&](uint32_t bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity));
    };
    if (ntiles > 0) {
      if (lane == 0) tc::mbar_arrive_expect_tx(BAR(kMQFull), C::kChunks * C::kQChunkBytes);
      __syncwarp();
      if (lane < C::kChunks)
        tc::tma_load_2d_(sbase + C::kOffQ + lane * C::kQChunkBytes, &q_map, BAR(kMQFull),
                         lane * 64, b * H + hg * C::kH);
    }
    int issued = 0;
    bool ok = true;
    int blk_next = ntiles > 0 ? tile_block(0) : -1;
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int st = j & 1;
      if (j >= 2 && !wait_all(BAR(kMKEmpty + st), ((j >> 1) - 1) & 1)) { ok = false; break; }
      const int blk = blk_next;
      blk_next = j + 1 < ntiles ? tile_block(j + 1) : -1;
      const uint32_t full = BAR(kMKFull + st);
      if (lane == 0) {
        if (blk < 0) record_error(err, PA_DEVERR_BLOCK_ID);
        tc::mbar_arrive_expect_tx(full, blk >= 0 ? C::kStageBytes : 0u);
      }
      __syncwarp();
      if (blk >= 0 && lane < C::kChunks)
        tc::tma_load_3d(sbase + C::kOffK + st * C::kStageBytes + lane * C::kKChunkBytes, &c_map,
                        full, lane * 64, (t0 + j * C::kBN) % bs, blk);
      issued = j + 1;
    }
    if (lane == 0) {
      if (!ok) fail();
      if (ntiles > 0 && !tc::mbar_wait(BAR(kMQFull), 0)) fail();
      for (int j = max(0, issued - 2); j < issued; ++j)
        if (!tc::mbar_wait(BAR(kMKFull + (j & 1)), (j >> 1) & 1)) fail();
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 mla_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = mla_encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_mla_tc(const void* q, const void* cache, const int32_t* block_table,
                          const int32_t* seq_lens, int B, int H, int bs, int num_blocks,
                          int max_blocks, float scale, int S, int chunk, float* ws, void* out,
                          float* lse, int* err, cudaStream_t stream) {
  using C = MlaTcCfg;
  CUtensorMap q_map, c_map;
  {
    const cuuint64_t dims[2] = {C::kDk, static_cast<cuuint64_t>(B) * H};
    const cuuint64_t strides[1] = {C::kDk * 2};
    const cuuint32_t box[2] = {64, C::kH};
    if (!encode(&q_map, q, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {C::kDk, static_cast<cuuint64_t>(bs),
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[2] = {C::kDk * 2, static_cast<cuuint64_t>(C::kDk) * 2 * bs};
    const cuuint32_t box[3] = {64, C::kBN, 1};
    if (!encode(&c_map, cache, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(mla_tc_kernel, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  dim3 grid(S, B, (H + C::kH - 1) / C::kH);
  mla_tc_kernel<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
      q_map, c_map, block_table, seq_lens, max_blocks, H, bs, num_blocks, scale * kLog2e, S,
      chunk, ws, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge(ws, B * H, S, C::kDv, out, lse, stream);
}

}  // namespace pa
