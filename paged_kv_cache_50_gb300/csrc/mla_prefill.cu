// MLA prefill in the multi-head formulation ("Attention Backends", section
// "Latent attention is a different cache, not just a different kernel":
// prefill and decode use different formulations of the same mathematics;
// "AttentionBackend: attention backend abstraction layer": forward_mha).
//
// Step 1 of 2, the expansion: every context token's latent c (kv_lora_rank
// 512) is multiplied by the model's kv_b_proj weight W [H][dn + dv][512],
// giving per head a key part k_nope = W[h][0:dn] c and a value
// v = W[h][dn:] c, stored as bf16 (the projection's output dtype) next to the
// token's k_pe:
//   K_ws[i][t][h] = [k_nope (dn) | k_pe (dr)]    [N][S_max][H][dn + dr]
//   V_ws[i][t][h] = v (dv)                       [N][S_max][H][dv]
// Step 2 (varlen_tc.cu, MLA mode) attends over K_ws / V_ws.
//
// GB300 design (a GEMM: 2 * 512 * H * (dn + dv) flops per token on the
// tcgen05 tensor cores): CTA = (128-token chunk, group of kMlaExpandHeads heads,
// request).  The chunk's 128 latent rows (128 KB, eight 64-column 128-byte
// swizzled slabs) are gathered once through the block table with TMA and
// stay resident; each head's 256 x 512 weight slice streams through a
// three-stage ring of 64-column slabs (32 KB each; two stages left the L2
// latency of a slab exposed: a slab feeds only 512 cycles of MMAs).  One
// thread issues
// D[128 x 256] = C W_h^T (M = 128 tokens, N = dn + dv = 256, K = 512) into one
// of two 256-column TMEM buffers, so the epilogue of head h (four warps, one
// token row per thread: TMEM -> bf16 -> global) overlaps the MMAs of head
// h + 1.  The epilogue writes each row with 32-byte stores: a warp's store
// touches 32 rows (one per thread), and whole sectors halve the store
// transactions against 16-byte ones.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_launch.h"
#include "tc_common.cuh"

namespace pa {

struct MlaExpCfg {
  static constexpr int kR = 512;            // kv_lora_rank
  static constexpr int kDr = 64;            // rope_dim
  static constexpr int kDn = 128;           // qk_nope_head_dim
  static constexpr int kDv = 128;           // v_head_dim
  static constexpr int kN = kDn + kDv;      // MMA N: one head's weight rows
  static constexpr int kM = 128;            // tokens per CTA
  static constexpr int kSlabs = kR / 64;    // 64-column (128-byte) slabs of the contraction
  static constexpr int kABytes = kM * kR * 2;           // 128 KB
  static constexpr int kASlab = kM * 128;               // 16 KB
  static constexpr int kWSlab = kN * 128;               // 32 KB
  static constexpr int kWStages = 3;
  static constexpr int kOffA = 0;
  static constexpr int kOffW = kABytes;
  static constexpr int kOffBar = kOffW + kWStages * kWSlab;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr int kThreads = 192;      // warp 0 MMA, 1 producer, 2-5 epilogue
  static constexpr uint32_t kTmemCols = 512;
};

enum MlaExpBar {
  kEAFull = 0,                                 // the latent tile has landed
  kEWFull = 1,                                 // [kWStages] weight slab stage
  kEWEmpty = kEWFull + MlaExpCfg::kWStages,    // [kWStages]
  kEDFull = kEWEmpty + MlaExpCfg::kWStages,    // [2] head accumulator buffer complete
  kEDEmpty = kEDFull + 2,                      // [2] buffer read out by the epilogue
  kEFinal = kEDEmpty + 2,
  kENumBars = kEFinal + 1
};

__global__ void __launch_bounds__(192, 1)
mla_expand_kernel(const __grid_constant__ CUtensorMap lat_map,
                  const __grid_constant__ CUtensorMap w_map,
                  const __nv_bfloat16* __restrict__ pool, const int32_t* __restrict__ block_table,
                  const int32_t* __restrict__ seq_lens, int max_blocks, int bs, int num_blocks,
                  int H, int heads_per_cta, int s_max, __nv_bfloat16* __restrict__ k_ws,
                  __nv_bfloat16* __restrict__ v_ws, int* err) {
  using C = MlaExpCfg;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  const int chunk = blockIdx.x, i = blockIdx.z;
  const int h0 = blockIdx.y * heads_per_cta;
  const int nh = min(heads_per_cta, H - h0);
  const int seq = seq_lens[i];
  const int t0 = chunk * C::kM;
  if (t0 >= seq || nh <= 0) return;
  const int rows = min(C::kM, seq - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks;
  const uint32_t bars = sbase + C::kOffBar;
  auto BAR = [&](int k) { return bars + 8u * static_cast<uint32_t>(k); };
  const uint32_t tmem_slot = bars + 8u * kENumBars;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + C::kOffBar + 8 * kENumBars + 8);
  auto fail = [&]() {
    *abort_flag = 1;
    record_error(err, PA_DEVERR_TIMEOUT);
  };

  if (threadIdx.x == 0) {
    tc::mbar_init(BAR(kEAFull), 1);
    for (int b = 0; b < C::kWStages; ++b) {
      tc::mbar_init(BAR(kEWFull + b), 1);
      tc::mbar_init(BAR(kEWEmpty + b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(BAR(kEDFull + b), 1);
      tc::mbar_init(BAR(kEDEmpty + b), 128);
    }
    tc::mbar_init(BAR(kEFinal), 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, C::kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + C::kOffBar + 8 * kENumBars);
  // Weight slabs in order: head j (0..nh-1), slab k (0..7) -> sequence n = j * 8 + k.
  const int n_slabs = nh * C::kSlabs;

  if (warp == 1) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::tma_prefetch_desc(&lat_map);
      tc::tma_prefetch_desc(&w_map);
    }
    // The latent tile: 16-token pieces (lane p < 8 owns piece p), eight
    // 64-column slabs each.  A piece past the request's end or with an
    // invalid block id is not loaded; its rows are zeroed below.
    const int p = lane;
    int blk = -1;
    bool load = false;
    if (p < C::kM / 16 && 16 * p < rows) {
      const int tok = t0 + 16 * p;
      const int idx = tok / bs;
      blk = idx < max_blocks ? __ldg(table + idx) : -1;
      load = blk >= 0 && blk < num_blocks;
      if (!load) record_error(err, PA_DEVERR_BLOCK_ID);
    }
    const unsigned loaded = __ballot_sync(0xffffffffu, load);
    if (lane == 0)
      tc::mbar_arrive_expect_tx(BAR(kEAFull),
                                static_cast<uint32_t>(__popc(loaded)) * C::kSlabs * 16 * 128);
    __syncwarp();
    if (load) {
      const int tok = t0 + 16 * p;
      for (int k = 0; k < C::kSlabs; ++k)
        tc::tma_load_3d(sbase + C::kOffA + k * C::kASlab + p * 16 * 128, &lat_map, BAR(kEAFull),
                        k * 64, tok % bs, blk);
    }
    // Weight slabs through the three-stage ring.
    if (lane == 0) {
      int issued = 0;
      for (int n = 0; n < n_slabs; ++n) {
        if (*abort_flag) break;
        const int st = n % C::kWStages;
        if (n >= C::kWStages &&
            !tc::mbar_wait(BAR(kEWEmpty + st), ((n / C::kWStages) - 1) & 1)) {
          fail();
          break;
        }
        const int h = h0 + n / C::kSlabs, k = n % C::kSlabs;
        tc::mbar_arrive_expect_tx(BAR(kEWFull + st), C::kWSlab);
        tc::tma_load_2d_(sbase + C::kOffW + st * C::kWSlab, &w_map, BAR(kEWFull + st), k * 64,
                         h * C::kN);
        issued = n + 1;
      }
      // No copy may still be landing when the CTA exits.
      if (!tc::mbar_wait(BAR(kEAFull), 0)) fail();
      for (int n = max(0, issued - C::kWStages); n < issued; ++n)
        if (!tc::mbar_wait(BAR(kEWFull + n % C::kWStages), (n / C::kWStages) & 1)) fail();
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ MMA issue
    // Rows of unloaded pieces must be finite: zero them before the first MMA
    // (the warp's 32 lanes cover a piece's 16 rows x 8 slabs x 8 chunks).
    {
      const unsigned missing = __ballot_sync(
          0xffffffffu, lane < C::kM / 16 && !(16 * lane < rows && [&] {
            const int idx = (t0 + 16 * lane) / bs;
            const int b = idx < max_blocks ? __ldg(table + idx) : -1;
            return b >= 0 && b < num_blocks;
          }()));
      for (int pz = 0; pz < C::kM / 16; ++pz) {
        if (!((missing >> pz) & 1u)) continue;
        for (int e = lane; e < 16 * C::kSlabs * 8; e += 32) {
          const int r = 16 * pz + (e >> 6), k = (e >> 3) & 7, c = e & 7;
          const uint32_t dst = sbase + C::kOffA + k * C::kASlab + (r >> 3) * 1024 + (r & 7) * 128 +
                               ((c ^ (r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
    }
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(C::kM, C::kN, 0, 0);
      bool ok = tc::mbar_wait(BAR(kEAFull), 0);
      if (!ok) fail();
      for (int j = 0; ok && j < nh; ++j) {
        const int b = j & 1;
        // Buffer b was last read out for head j - 2.
        if (j >= 2 && !tc::mbar_wait(BAR(kEDEmpty + b), ((j >> 1) - 1) & 1)) {
          fail();
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int k = 0; k < C::kSlabs; ++k) {
          const int n = j * C::kSlabs + k, st = n % C::kWStages;
          if (*abort_flag || !tc::mbar_wait(BAR(kEWFull + st), (n / C::kWStages) & 1)) {
            fail();
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a = sbase + C::kOffA + k * C::kASlab;
          const uint32_t w = sbase + C::kOffW + st * C::kWSlab;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_bf16_ss(tmem + b * 256, tc::smem_desc_sw128(a + kk * 32, 16, 1024),
                            tc::smem_desc_sw128(w + kk * 32, 16, 1024), idesc,
                            (k > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit(BAR(kEWEmpty + st));   // the slab stage is free once these complete
        }
        if (ok) tc::mma_commit(BAR(kEDFull + b));
      }
      tc::mma_commit(BAR(kEFinal));
      if (!tc::mbar_wait(BAR(kEFinal), 0)) fail();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                  // TMEM lane quarter of this warp
    const int t = q * 32 + lane;             // token row of the tile
    const bool valid = t < rows;
    const int64_t tok = static_cast<int64_t>(i) * s_max + t0 + t;
    // This token's k_pe, copied next to every head's k_nope.
    uint4 kpe[C::kDr / 8];
    {
      const int idx = (t0 + t) / bs;
      const int b = valid && idx < max_blocks ? __ldg(table + idx) : -1;
      const bool ok = b >= 0 && b < num_blocks;
      const uint4* src = reinterpret_cast<const uint4*>(
          pool + (static_cast<int64_t>(ok ? b : 0) * bs + (t0 + t) % bs) * (C::kR + C::kDr) + C::kR);
#pragma unroll
      for (int c = 0; c < C::kDr / 8; ++c) kpe[c] = ok ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
    }
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    for (int j = 0; j < nh; ++j) {
      const int b = j & 1, h = h0 + j;
      const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(BAR(kEDFull + b), (j >> 1) & 1));
      if (!ok) {
        if (lane == 0) fail();
        break;
      }
      tc::tc_fence_after();
      // 32-byte stores (one whole sector each): the thread's row is 384 bytes
      // of K (k_nope | k_pe) and 256 of V, both 32-byte aligned.
      uint32_t* kdst = reinterpret_cast<uint32_t*>(k_ws + (tok * H + h) * (C::kDn + C::kDr));
      uint32_t* vdst = reinterpret_cast<uint32_t*>(v_ws + (tok * H + h) * C::kDv);
#pragma unroll
      for (int c2 = 0; c2 < C::kN / 64; ++c2) {
        uint32_t r[2][32];
        tc::tmem_ld32(tmem + lane_base + b * 256 + c2 * 64, r[0]);
        tc::tmem_ld32(tmem + lane_base + b * 256 + c2 * 64 + 32, r[1]);
        tc::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = 2 * c2 + u;   // 32 columns: 64 bytes of bf16
            uint32_t* dst = c < C::kDn / 32 ? kdst + c * 16 : vdst + (c - C::kDn / 32) * 16;
#pragma unroll
            for (int v = 0; v < 2; ++v) {
              uint32_t w[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w[e] = pack_bf16(__uint_as_float(r[u][v * 16 + 2 * e]),
                                 __uint_as_float(r[u][v * 16 + 2 * e + 1]));
              st_global_v8(dst + v * 8, w);
            }
          }
        }
      }
      if (valid) {
#pragma unroll
        for (int c = 0; c < C::kDr / 16; ++c) {
          const uint32_t w[8] = {kpe[2 * c].x, kpe[2 * c].y, kpe[2 * c].z, kpe[2 * c].w,
                                 kpe[2 * c + 1].x, kpe[2 * c + 1].y, kpe[2 * c + 1].z,
                                 kpe[2 * c + 1].w};
          st_global_v8(kdst + C::kDn / 2 + c * 8, w);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(BAR(kEDEmpty + b));
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

// Latent pool [nb][bs][576] viewed 3-D (innermost first): 64-column x
// 16-token boxes, 128-byte swizzle.
bool make_latent_map(CUtensorMap* map, const void* pool, int nb, int bs) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {576, static_cast<cuuint64_t>(bs), static_cast<cuuint64_t>(nb)};
  const cuuint64_t strides[2] = {576 * 2, static_cast<cuuint64_t>(bs) * 576 * 2};
  const cuuint32_t box[3] = {64, 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// kv_b_proj weight [H * 256][512] viewed 2-D: 64-column x 256-row boxes.
bool make_weight_map(CUtensorMap* map, const void* w, int H) {
  auto fn = tensor_map_encoder();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {512, static_cast<cuuint64_t>(H) * 256};
  const cuuint64_t strides[1] = {512 * 2};
  const cuuint32_t box[2] = {64, 256};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Heads per CTA of the expansion: a CTA reuses its resident latent tile for
// this many heads' weight slices.
constexpr int kMlaExpandHeads = 16;
cudaError_t launch_mla_expand(const void* pool, const void* w_kv_b, const int32_t* block_table,
                              const int32_t* seq_lens, int N, int H, int bs, int num_blocks,
                              int max_blocks, int max_seq_len, int s_max, void* k_ws, void* v_ws,
                              int* err, cudaStream_t stream) {
  using C = MlaExpCfg;
  CUtensorMap lat, wm;
  if (!make_latent_map(&lat, pool, num_blocks, bs) || !make_weight_map(&wm, w_kv_b, H))
    return cudaErrorInvalidValue;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(mla_expand_kernel, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  const int chunks = (max_seq_len + C::kM - 1) / C::kM;
  if (chunks == 0 || N == 0) return cudaSuccess;
  const dim3 grid(chunks, (H + kMlaExpandHeads - 1) / kMlaExpandHeads, N);
  mla_expand_kernel<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
      lat, wm, static_cast<const __nv_bfloat16*>(pool), block_table, seq_lens, max_blocks, bs,
      num_blocks, H, kMlaExpandHeads, s_max, static_cast<__nv_bfloat16*>(k_ws),
      static_cast<__nv_bfloat16*>(v_ws), err);
  return cudaGetLastError();
}

}  // namespace pa
