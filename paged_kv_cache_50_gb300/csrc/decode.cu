// Split-KV decode, stage 1, for the standard paged layout
// [num_blocks, 2, block_size, Hkv, d] (stage 2, the LSE merge, is merge.cu).
//
// Method: "Chapter 1: attention backends" (zero-to-sglang), section 3.1 --
// a decode query has too little parallelism, so the context is split along
// the sequence, each split yields a partial output with its softmax
// normaliser, and the partials are merged; section 4.1 -- inside a split the
// keys are consumed tile by tile with an online softmax (running max and sum,
// earlier output rescaled when the max grows, Fig. 5c).  Workspace layout
// [N, Hq, S, d + 1] with the LSE in the last slot: data-flow section of
// "Triton and MLA" (vllm-arch-zh).
//
// GB300 design (decode is HBM-bound: every K/V byte is read exactly once):
//  * one CTA per (split, kv head, request); its 4 warps take the split's
//    16-token sub-blocks round-robin, each warp with its own cp.async
//    pipeline (STAGES deep) into an XOR-swizzled shared-memory ring, so the
//    main loop has no CTA-wide barrier;
//  * the 16 tokens of a sub-block are the M dimension of mma.m16n8k16 and
//    the Hq/Hkv query heads of the kv group its N dimension (8 per n-tile),
//    so the K/V bytes fetched once serve the whole group: S^T = K Q^T with K
//    read by ldmatrix as the A operand, online softmax in registers (exp2
//    with the scale folded in; per head over the tokens, i.e. across lanes),
//    then O^T += V^T P^T with V^T read by ldmatrix.trans and P^T gathered by
//    four shuffles of bf16 pairs -- d/16 MMAs per product per sub-block and
//    d/16 x 4 output registers per n-tile;
//  * the running max moves only when a sub-block's max exceeds it by more
//    than 8 (log2 units), so the output rescale is rare; the next block id is
//    loaded one iteration before its copies are issued;
//  * the four warps' (max, sum, O) states are merged through shared memory
//    at the end and the split's normalised partial and natural-log LSE are
//    written to the workspace.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int STAGES, int NT>
struct DecodeCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRowBytes = D * 2;            // one token of one head
  static constexpr int kChunks = D / 8;              // 16-byte chunks per row
  static constexpr int kTileBytes = 16 * kRowBytes;  // 16 tokens of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes; // K + V
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static constexpr int kPipeBytes = kWarps * kWarpBytes;
  // Combine buffer: per warp 8*NT head rows of d floats, kOStride apart
  // (= 4 mod 32: the fragment stores hit 32 distinct banks).
  static constexpr int kOStride = D + 4;
  static constexpr int kHeads = 8 * NT;
  static constexpr int kCombineBytes = kWarps * (kHeads * kOStride + 3 * kHeads) * 4;
  static constexpr int kSmemBytes = kPipeBytes > kCombineBytes ? kPipeBytes : kCombineBytes;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

template <int D, int STAGES, int NT>
__global__ void __launch_bounds__(128)
decode_splitkv_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ cache,
                      const int32_t* __restrict__ block_table, const int32_t* __restrict__ seq_lens,
                      int max_blocks, int Hq, int Hkv, int bs, int bs_log2, int num_blocks, float scale_log2,
                      int S, int chunk, float* __restrict__ ws, int* err, DecodeExt ext) {
  using C = DecodeCfg<D, STAGES, NT>;
  constexpr int kK = D / 16;   // k-steps of K Q^T = d-tiles of V^T P^T
  constexpr float kRescale = 8.f;
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int grp = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;

  // Every input may come from the previous kernel in the stream.
  pdl_wait();
  // Split s covers [s*chunk, (s+1)*chunk) of the request (the last split runs
  // to the end), chunk being one block-aligned size for the whole batch.
  const long long a0 = static_cast<long long>(s) * chunk;
  // ext.seq_off tokens at the front of every request are skipped (their
  // blocks are the first ext.table_col0 columns of the table row).
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks + ext.table_col0;
  const int cols = max_blocks - ext.table_col0;
  // Block ids of the warp's first STAGES sub-blocks, read together with
  // seq_len (they do not depend on it when the split is not empty, which
  // then starts at a0); ids of sub-blocks the split does not have are never
  // used.
  int first_blk[STAGES];
#pragma unroll
  for (int n = 0; n < STAGES; ++n) {
    const long long tok = a0 + (warp + n * C::kWarps) * 16;
    const long long col = bs_log2 >= 0 ? tok >> bs_log2 : tok / bs;
    first_blk[n] = col < cols ? block_at(table, static_cast<int>(col), cols) : -1;
  }
  const int seq = max(0, seq_lens[i] - ext.seq_off);
  const int t0 = static_cast<int>(a0 < seq ? a0 : seq);
  const int t1 = (s == S - 1) ? seq : static_cast<int>(a0 + chunk < seq ? a0 + chunk : seq);
  const int nsb = (t1 - t0 + 15) >> 4;
  if (nsb == 0) {
    // An empty split (the request ends before it starts): o = 0, lse = -inf
    // for the group's heads, and nothing else.  With the split size taken
    // from the batch's longest request, many of a ragged batch's splits are
    // empty.
    pdl_trigger();
    for (int idx = threadIdx.x; idx < grp * (D + 1); idx += C::kThreads) {
      const int r = idx / (D + 1), e = idx - r * (D + 1);
      ws[((static_cast<int64_t>(i) * Hq + kvh * grp + r) * ext.ws_slots + ext.ws_slot0 + s) *
             (D + 1) + e] = e == D ? -CUDART_INF_F : 0.f;
    }
    return;
  }
  const int my_n = nsb > warp ? (nsb - warp + C::kWarps - 1) / C::kWarps : 0;

  // Q^T as the B operand: lane (gid, tid4) holds head nt*8 + gid (zero past
  // the group), dimensions 16 kk + 2 tid4 + {0, 1} and + {8, 9}.
  uint32_t qf[NT][kK][2];
  {
    const __nv_bfloat16* qb = q + (static_cast<int64_t>(i) * Hq + static_cast<int64_t>(kvh) * grp) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + gid;
      const bool ok = h < grp;
#pragma unroll
      for (int kk = 0; kk < kK; ++kk) {
        qf[nt][kk][0] = ok ? ld_u32(qb + h * D + kk * 16 + 2 * tid4) : 0u;
        qf[nt][kk][1] = ok ? ld_u32(qb + h * D + kk * 16 + 8 + 2 * tid4) : 0u;
      }
    }
  }

  const uint32_t wbase = smem_u32(smem) + warp * C::kWarpBytes;
  const int64_t row_stride = static_cast<int64_t>(Hkv) * D;

  // Block id of the warp's n-th sub-block (loaded one iteration before its
  // copies are issued, so the table read is off the critical path).
  auto lookup = [&](int n) {
    return block_at(table, div_bs(t0 + (warp + n * C::kWarps) * 16, bs, bs_log2), cols);
  };
  // Bit n % 32 of okbits: the n-th sub-block's block id was valid (at most
  // STAGES sub-blocks are between issue and use).
  uint32_t okbits = 0;
  auto issue = [&](int n, int blk) {
    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const bool ok = blk >= 0 && blk < num_blocks;
    if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID);
    okbits = (okbits & ~(1u << (n & 31))) | (static_cast<uint32_t>(ok) << (n & 31));
    const int off = mod_bs(tb, bs, bs_log2);
    const __nv_bfloat16* kbase =
        cache + ((static_cast<int64_t>(ok ? blk : 0) * 2) * bs + off) * row_stride +
        static_cast<int64_t>(kvh) * D;
    const __nv_bfloat16* vbase = kbase + static_cast<int64_t>(bs) * row_stride;
    const uint32_t kdst = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
    for (int k = 0; k < 16 * C::kChunks / 32; ++k) {
      const int c = lane + 32 * k;
      const int r = c / C::kChunks, cc = c % C::kChunks;
      const int bytes = (ok && tb + r < t1) ? 16 : 0;
      const uint32_t so = swz(r, cc, C::kRowBytes);
      cp_async_16(kdst + so, kbase + r * row_stride + cc * 8, bytes);
      cp_async_16(vdst + so, vbase + r * row_stride + cc * 8, bytes);
    }
  };

  // Per lane: heads nt*8 + 2 tid4 + j (j = 0, 1) -- running max (replicated
  // over the 8 token lanes), partial sums over the lane's tokens, and O^T.
  // l_r: the weights' sums (for the LSE); lb_r: the sums of the weights
  // rounded to bf16, as the PV product multiplies them (the output divisor).
  float m_r[NT][2], l_r[NT][2], lb_r[NT][2];
  float o[NT][kK][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_r[nt][0] = m_r[nt][1] = -CUDART_INF_F;
    l_r[nt][0] = l_r[nt][1] = 0.f;
    lb_r[nt][0] = lb_r[nt][1] = 0.f;
#pragma unroll
    for (int md = 0; md < kK; ++md) o[nt][md][0] = o[nt][md][1] = o[nt][md][2] = o[nt][md][3] = 0.f;
  }

#pragma unroll
  for (int n = 0; n < STAGES - 1; ++n) {
    if (n < my_n) issue(n, first_blk[n]);
    cp_async_commit();
  }
  int next_blk = STAGES - 1 < my_n ? first_blk[STAGES - 1] : -1;

  // Source lanes of the P^T operand: tokens 2 tid4 (srcA) and 2 tid4 + 1
  // (srcB) hold head gid in the lane of tid4' = gid / 2, half gid % 2.
  const int srcA = 8 * tid4 + (gid >> 1), srcB = srcA + 4;
  const uint32_t psel = (gid & 1) ? 0x7632u : 0x5410u;
  // ldmatrix row addresses: K as A (token lane & 15, half lane >> 4 of the
  // k-step), V^T as A (token (lane & 7) + 8 (lane >> 4), half (lane >> 3) & 1).
  const int k_row = lane & 15, k_half = lane >> 4;
  const int v_row = (lane & 7) + ((lane >> 4) << 3), v_half = (lane >> 3) & 1;

  for (int n = 0; n < my_n; ++n) {
    cp_async_wait<STAGES - 2>();
    __syncwarp();
    if (n + STAGES - 1 < my_n) {
      issue(n + STAGES - 1, next_blk);
      if (n + STAGES < my_n) next_blk = lookup(n + STAGES);
    }
    cp_async_commit();

    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const int lim = ((okbits >> (n & 31)) & 1u) ? min(16, t1 - tb) : 0;
    const uint32_t kb = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;

    // S^T = K Q^T: rows = tokens gid, gid + 8; columns = heads.  Even and
    // odd k-steps go to separate accumulators (two MMA chains of half the
    // length).
    float sc[NT][4];
    {
      float s2[NT][2][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) s2[nt][h][0] = s2[nt][h][1] = s2[nt][h][2] = s2[nt][h][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < kK; ++kk) {
        uint32_t a[4];
        ldmatrix_x4(kb + swz(k_row, 2 * kk + k_half, C::kRowBytes), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_bf16_16816(s2[nt][kk & 1], a, qf[nt][kk][0], qf[nt][kk][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = s2[nt][0][e] + s2[nt][1][e];
    }

    // Online softmax (log2 domain, scale folded in), per head over the 16
    // tokens: two in the lane, the rest across the 8 token lanes.  The
    // reference max moves only when a sub-block's max exceeds it by more than
    // kRescale, so the output rescale is rare and the weights stay < 2^8.
    const bool v0 = gid < lim, v1 = gid + 8 < lim;
    uint32_t pb[NT][2];   // P^T operand: b0 (tokens 2 tid4, +1), b1 (+8, +9)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float x0 = v0 ? sc[nt][j] * scale_log2 : -CUDART_INF_F;
        const float x1 = v1 ? sc[nt][2 + j] * scale_log2 : -CUDART_INF_F;
        float mx = fmaxf(x0, x1);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (mx > m_r[nt][j] + kRescale) {
          const float alpha = fast_exp2(m_r[nt][j] - mx);   // 0 when m_r = -inf
          m_r[nt][j] = mx;
          l_r[nt][j] *= alpha;
          lb_r[nt][j] *= alpha;
#pragma unroll
          for (int md = 0; md < kK; ++md) {
            o[nt][md][j] *= alpha;
            o[nt][md][2 + j] *= alpha;
          }
        }
        const float mu = m_r[nt][j] == -CUDART_INF_F ? 0.f : m_r[nt][j];
        p[j] = fast_exp2(x0 - mu);
        p[2 + j] = fast_exp2(x1 - mu);
        l_r[nt][j] += p[j] + p[2 + j];
      }
      // S^T -> P^T: this lane's (token, head pair) values as bf16 pairs, then
      // each lane gathers its head's four tokens.
      const uint32_t u_lo = pack_bf16(p[0], p[1]);   // token gid, heads 2 tid4, +1
      const uint32_t u_hi = pack_bf16(p[2], p[3]);   // token gid + 8
      add_bf16x2_f32(lb_r[nt][0], lb_r[nt][1], u_lo);
      add_bf16x2_f32(lb_r[nt][0], lb_r[nt][1], u_hi);
      const uint32_t xa = __shfl_sync(0xffffffffu, u_lo, srcA);
      const uint32_t xb = __shfl_sync(0xffffffffu, u_lo, srcB);
      const uint32_t ya = __shfl_sync(0xffffffffu, u_hi, srcA);
      const uint32_t yb = __shfl_sync(0xffffffffu, u_hi, srcB);
      pb[nt][0] = __byte_perm(xa, xb, psel);
      pb[nt][1] = __byte_perm(ya, yb, psel);
    }

    // O^T += V^T P^T, V^T tiles read transposed from the token-major V tile.
#pragma unroll
    for (int md = 0; md < kK; ++md) {
      uint32_t a[4];
      ldmatrix_x4_trans(vb + swz(v_row, 2 * md + v_half, C::kRowBytes), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[nt][md], a, pb[nt][0], pb[nt][1]);
    }
  }
  cp_async_wait<0>();
  // The merge may start launching (it waits for this kernel to complete).
  pdl_trigger();

  // Partial sums over the 8 token lanes.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 4);
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 8);
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 16);
      lb_r[nt][j] += __shfl_xor_sync(0xffffffffu, lb_r[nt][j], 4);
      lb_r[nt][j] += __shfl_xor_sync(0xffffffffu, lb_r[nt][j], 8);
      lb_r[nt][j] += __shfl_xor_sync(0xffffffffu, lb_r[nt][j], 16);
    }

  // Merge the four warps' states through shared memory.
  __syncthreads();
  float* cbuf = reinterpret_cast<float*>(smem);
  float* mbuf = cbuf + C::kWarps * C::kHeads * C::kOStride;  // [warp][kHeads]
  float* lbuf = mbuf + C::kWarps * C::kHeads;
  float* rbuf = lbuf + C::kWarps * C::kHeads;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int md = 0; md < kK; ++md)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = nt * 8 + 2 * tid4 + (e & 1);
        cbuf[(warp * C::kHeads + h) * C::kOStride + md * 16 + gid + 8 * (e >> 1)] = o[nt][md][e];
      }
    if (gid == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mbuf[warp * C::kHeads + nt * 8 + 2 * tid4 + j] = m_r[nt][j];
        lbuf[warp * C::kHeads + nt * 8 + 2 * tid4 + j] = l_r[nt][j];
        rbuf[warp * C::kHeads + nt * 8 + 2 * tid4 + j] = lb_r[nt][j];
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * D; idx += C::kThreads) {
    const int r = idx / D, e = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mbuf[w * C::kHeads + r]);
    float* dst =
        ws + ((static_cast<int64_t>(i) * Hq + kvh * grp + r) * ext.ws_slots + ext.ws_slot0 + s) * (D + 1);
    if (M == -CUDART_INF_F) {
      dst[e] = 0.f;
      if (e == 0) dst[D] = -CUDART_INF_F;
      continue;
    }
    float L = 0.f, LB = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float f = fast_exp2(mbuf[w * C::kHeads + r] - M);
      L += f * lbuf[w * C::kHeads + r];
      LB += f * rbuf[w * C::kHeads + r];
      acc += f * cbuf[(w * C::kHeads + r) * C::kOStride + e];
    }
    dst[e] = acc / LB;
    if (e == 0) dst[D] = (M + log2f(L)) * kLn2;
  }
}

template <int D, int STAGES, int NT>
static cudaError_t launch_decode_t(const void* q, const void* cache, const int32_t* block_table,
                                   const int32_t* seq_lens, int N, int Hq, int Hkv, int bs,
                                   int num_blocks, int max_blocks, float scale, int S, int chunk,
                                   float* ws, int* err, const DecodeExt& ext,
                                   cudaStream_t stream) {
  using C = DecodeCfg<D, STAGES, NT>;
  auto kern = decode_splitkv_kernel<D, STAGES, NT>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(S, Hkv, N), dim3(C::kThreads), C::kSmemBytes, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(cache),
                    block_table, seq_lens, max_blocks, Hq, Hkv, bs, block_size_log2(bs), num_blocks,
                    scale * kLog2e, S,
                    chunk, ws, err, ext);
}

cudaError_t launch_decode_splitkv(const void* q, const void* cache, const int32_t* block_table,
                                  const int32_t* seq_lens, int N, int Hq, int Hkv, int d, int bs,
                                  int num_blocks, int max_blocks, float scale, int S, int chunk,
                                  float* ws, int* err, cudaStream_t stream, const DecodeExt* ext) {
  const DecodeExt plain{0, 0, S, 0};
  const DecodeExt& x = ext != nullptr ? *ext : plain;
  const bool wide = Hq / Hkv > 8;   // groups of 9..16 heads take two n-tiles
#define PA_DECODE_LAUNCH(DD, ST, NTT)                                                          \
  return launch_decode_t<DD, ST, NTT>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs,         \
                                      num_blocks, max_blocks, scale, S, chunk, ws, err, x, stream)
  if (d == 128) {
    if (wide) PA_DECODE_LAUNCH(128, 2, 2);
    PA_DECODE_LAUNCH(128, 2, 1);
  }
  if (wide) PA_DECODE_LAUNCH(64, 4, 2);
  PA_DECODE_LAUNCH(64, 4, 1);
#undef PA_DECODE_LAUNCH
}

}  // namespace pa
