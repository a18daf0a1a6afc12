// Split-KV decode (stage 1) over an fp8 pool of e4m3 codes,
// [num_blocks, 2, block_size, Hkv, d] bytes.  An entry stands for its e4m3
// value times the layer's k_scale (K half) or v_scale (V half): "Triton and
// MLA" (vllm-arch-zh), data flow -- the decode kernel always receives both
// scales.  The split, the online softmax and the workspace layout
// [N, Hq, S, d + 1] are those of the bf16 stage 1 ("Chapter 1: attention
// backends", sections 3.1 and 4.1); the LSE merge is shared.
//
// GB300 design (HBM-bound; an fp8 pool halves the bytes per token):
//  * one CTA per (split, kv head, request), four warps taking 16-token
//    sub-blocks round-robin, each warp with its own cp.async ring of raw code
//    tiles (no CTA-wide barrier in the main loop);
//  * codes go from shared memory straight into mma.m16n8k16 operand
//    registers: e4m3 -> f16 is exact (cvt.rn.f16x2.e4m3x2), so the MMAs run
//    on f16 operands with Q converted bf16 -> f16 once (exact for |q| in
//    f16's normal range) and P packed as f16;
//  * a dot product does not depend on the order of its terms, so the head
//    dimension is permuted alike in Q and K: the 4 k-values a lane owns in
//    k-step kk are the bytes [tid4 * d/4 + 4 kk, + 4) of its token's row,
//    one 32-bit word of codes;
//  * the output columns are permuted too: column n of the MMA's n-tile nd is
//    head dimension n * d/8 + nd, so a lane's V operand bytes are d/8
//    contiguous codes of each of its four token rows, paired across rows with
//    byte permutes; the combine writes the columns back in order;
//  * k_scale folds into the exp2 scale and v_scale into the partial output
//    (the LSE does not depend on V).
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int STAGES>
struct DecodeFp8Cfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunks = D / 16;             // 16-byte chunks per row
  static constexpr int kTileBytes = 16 * D;          // 16 tokens of K (or V) codes
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static constexpr int kPipeBytes = kWarps * kWarpBytes;
  static constexpr int kOStride = D + 4;
  static constexpr int kCombineBytes = kWarps * (16 * kOStride + 32) * 4;
  static constexpr int kSmemBytes = kPipeBytes > kCombineBytes ? kPipeBytes : kCombineBytes;
};

// Byte offset of 16-byte chunk c of token row r in a code tile.  The XOR
// keeps both read patterns free of bank conflicts: the K reads (8 lanes = 2
// rows x 4 chunks of one parity) and the V reads (8 lanes = 4 rows of one
// parity x 2 chunks) for d = 128; for d = 64 two rows share a 128-byte line.
template <int D>
__device__ __forceinline__ uint32_t swz8(int r, int c) {
  if constexpr (D == 128)
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
  else
    return static_cast<uint32_t>(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}

// Four e4m3 codes (byte 0 lowest) -> two f16x2 words (codes 0,1 and 2,3,
// the lower code in the low half).  Exact.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two consecutive bf16 of q as one f16x2 word.
__device__ __forceinline__ uint32_t q_pair_f16(const __nv_bfloat16* p) {
  const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
  const float2 f = __bfloat1622float2(v);
  return pack_f16(f.x, f.y);
}

template <int D, int STAGES>
__global__ void __launch_bounds__(128)
decode_splitkv_fp8_kernel(const __nv_bfloat16* __restrict__ q, const uint8_t* __restrict__ cache,
                          const int32_t* __restrict__ block_table,
                          const int32_t* __restrict__ seq_lens, int max_blocks, int Hq, int Hkv,
                          int bs, int num_blocks, float scale_log2, float v_scale, int S,
                          int chunk, float* __restrict__ ws, int* err) {
  using C = DecodeFp8Cfg<D, STAGES>;
  constexpr int kW = D / 32;  // 32-bit words of V codes per lane per token row
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int grp = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;

  pdl_wait();
  const int seq = seq_lens[i];
  const long long a0 = static_cast<long long>(s) * chunk;
  const int t0 = static_cast<int>(a0 < seq ? a0 : seq);
  const int t1 = (s == S - 1) ? seq : static_cast<int>(a0 + chunk < seq ? a0 + chunk : seq);
  const int nsb = (t1 - t0 + 15) >> 4;
  const int my_n = nsb > warp ? (nsb - warp + C::kWarps - 1) / C::kWarps : 0;

  // Q of the kv group as the A operand (rows = the group's heads, zero-padded
  // to 16), head dimension in the permuted order described above.
  uint32_t qf[D / 16][4];
  {
    const __nv_bfloat16* qb = q + (static_cast<int64_t>(i) * Hq + static_cast<int64_t>(kvh) * grp) * D;
    const bool r0 = gid < grp, r1 = gid + 8 < grp;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c0 = tid4 * (D / 4) + kk * 4;
      qf[kk][0] = r0 ? q_pair_f16(qb + gid * D + c0) : 0u;
      qf[kk][1] = r1 ? q_pair_f16(qb + (gid + 8) * D + c0) : 0u;
      qf[kk][2] = r0 ? q_pair_f16(qb + gid * D + c0 + 2) : 0u;
      qf[kk][3] = r1 ? q_pair_f16(qb + (gid + 8) * D + c0 + 2) : 0u;
    }
  }

  const uint32_t wbase = smem_u32(smem) + warp * C::kWarpBytes;
  const int64_t row_stride = static_cast<int64_t>(Hkv) * D;  // bytes per token row
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks;

  auto issue = [&](int n) {
    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const int blk = block_at(table, tb / bs, max_blocks);
    const bool ok = blk >= 0 && blk < num_blocks;
    if (!ok && lane == 0) record_error(err, PA_DEVERR_BLOCK_ID);
    const int off = tb % bs;
    const uint8_t* kbase = cache + ((static_cast<int64_t>(ok ? blk : 0) * 2) * bs + off) * row_stride +
                           static_cast<int64_t>(kvh) * D;
    const uint8_t* vbase = kbase + static_cast<int64_t>(bs) * row_stride;
    const uint32_t kdst = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
    for (int k = 0; k < 16 * C::kChunks / 32; ++k) {
      const int c = lane + 32 * k;
      const int r = c / C::kChunks, cc = c % C::kChunks;
      const int bytes = (ok && tb + r < t1) ? 16 : 0;
      const uint32_t so = swz8<D>(r, cc);
      cp_async_16(kdst + so, kbase + r * row_stride + cc * 16, bytes);
      cp_async_16(vdst + so, vbase + r * row_stride + cc * 16, bytes);
    }
  };

  float m_r[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_r[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

#pragma unroll
  for (int n = 0; n < STAGES - 1; ++n) {
    if (n < my_n) issue(n);
    cp_async_commit();
  }

  for (int n = 0; n < my_n; ++n) {
    cp_async_wait<STAGES - 2>();
    __syncwarp();
    if (n + STAGES - 1 < my_n) issue(n + STAGES - 1);
    cp_async_commit();

    const int tb = t0 + (warp + n * C::kWarps) * 16;
    const int blk = block_at(table, tb / bs, max_blocks);
    const int lim = (blk >= 0 && blk < num_blocks) ? min(16, t1 - tb) : 0;
    const uint32_t kb = wbase + (n % STAGES) * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;

    // S = Q K^T: 16 heads x 16 tokens; lane's B operand = token nt*8 + gid.
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int r = nt * 8 + gid;
      uint32_t kw[D / 16];
      if constexpr (D == 128) {
        const uint4 x0 = lds128(kb + swz8<D>(r, 2 * tid4));
        const uint4 x1 = lds128(kb + swz8<D>(r, 2 * tid4 + 1));
        kw[0] = x0.x; kw[1] = x0.y; kw[2] = x0.z; kw[3] = x0.w;
        kw[4] = x1.x; kw[5] = x1.y; kw[6] = x1.z; kw[7] = x1.w;
      } else {
        const uint4 x0 = lds128(kb + swz8<D>(r, tid4));
        kw[0] = x0.x; kw[1] = x0.y; kw[2] = x0.z; kw[3] = x0.w;
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t b0, b1;
        e4m3x4_to_f16(kw[kk], b0, b1);
        mma_f16_16816(sc[nt], qf[kk], b0, b1);
      }
    }

    // Online softmax (log2 domain, scale * k_scale folded in).
    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = nt * 8 + 2 * tid4 + (e & 1);
        const float x = tok < lim ? sc[nt][e] * scale_log2 : -CUDART_INF_F;
        sc[nt][e] = x;
        mx[e >> 1] = fmaxf(mx[e >> 1], x);
      }
    float alpha[2], mu[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m_r[r], mx[r]);
      mu[r] = mn == -CUDART_INF_F ? 0.f : mn;
      alpha[r] = fast_exp2(m_r[r] - mu[r]);
      m_r[r] = mn;
      l_r[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = fast_exp2(sc[nt][e] - mu[e >> 1]);
        sc[nt][e] = p;
        l_r[e >> 1] += p;
      }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= alpha[0];
      o[nd][1] *= alpha[0];
      o[nd][2] *= alpha[1];
      o[nd][3] *= alpha[1];
    }
    uint32_t pf[4];
    pf[0] = pack_f16(sc[0][0], sc[0][1]);
    pf[1] = pack_f16(sc[0][2], sc[0][3]);
    pf[2] = pack_f16(sc[1][0], sc[1][1]);
    pf[3] = pack_f16(sc[1][2], sc[1][3]);

    // O += P V.  The lane's B operands are tokens 2 tid4 + {0, 1} (b0) and
    // 2 tid4 + {8, 9} (b1) of head dimension gid * d/8 + nd.
    {
      uint32_t va[kW], vb1[kW], vc[kW], ve[kW];
      const int rA = 2 * tid4;
      if constexpr (D == 128) {
        const uint4 xa = lds128(vb + swz8<D>(rA, gid)), xb = lds128(vb + swz8<D>(rA + 1, gid));
        const uint4 xc = lds128(vb + swz8<D>(rA + 8, gid)), xe = lds128(vb + swz8<D>(rA + 9, gid));
        va[0] = xa.x; va[1] = xa.y; va[2] = xa.z; va[3] = xa.w;
        vb1[0] = xb.x; vb1[1] = xb.y; vb1[2] = xb.z; vb1[3] = xb.w;
        vc[0] = xc.x; vc[1] = xc.y; vc[2] = xc.z; vc[3] = xc.w;
        ve[0] = xe.x; ve[1] = xe.y; ve[2] = xe.z; ve[3] = xe.w;
      } else {
        const uint32_t h = (gid & 1) * 8;
        const uint2 xa = lds64(vb + swz8<D>(rA, gid >> 1) + h);
        const uint2 xb = lds64(vb + swz8<D>(rA + 1, gid >> 1) + h);
        const uint2 xc = lds64(vb + swz8<D>(rA + 8, gid >> 1) + h);
        const uint2 xe = lds64(vb + swz8<D>(rA + 9, gid >> 1) + h);
        va[0] = xa.x; va[1] = xa.y;
        vb1[0] = xb.x; vb1[1] = xb.y;
        vc[0] = xc.x; vc[1] = xc.y;
        ve[0] = xe.x; ve[1] = xe.y;
      }
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        uint32_t b0[4], b1[4];
        e4m3x4_to_f16(__byte_perm(va[w], vb1[w], 0x5140), b0[0], b0[1]);
        e4m3x4_to_f16(__byte_perm(va[w], vb1[w], 0x7362), b0[2], b0[3]);
        e4m3x4_to_f16(__byte_perm(vc[w], ve[w], 0x5140), b1[0], b1[1]);
        e4m3x4_to_f16(__byte_perm(vc[w], ve[w], 0x7362), b1[2], b1[3]);
#pragma unroll
        for (int j = 0; j < 4; ++j) mma_f16_16816(o[4 * w + j], pf, b0[j], b1[j]);
      }
    }
  }
  cp_async_wait<0>();
  pdl_trigger();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }

  // Merge the four warps' states through shared memory, putting the output
  // columns back in head-dimension order.
  __syncthreads();
  float* cbuf = reinterpret_cast<float*>(smem);
  float* mbuf = cbuf + C::kWarps * 16 * C::kOStride;
  float* lbuf = mbuf + C::kWarps * 16;
  {
    float* ob = cbuf + warp * 16 * C::kOStride;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const int c0 = (2 * tid4) * (D / 8) + nd, c1 = c0 + D / 8;
      ob[gid * C::kOStride + c0] = o[nd][0];
      ob[gid * C::kOStride + c1] = o[nd][1];
      ob[(gid + 8) * C::kOStride + c0] = o[nd][2];
      ob[(gid + 8) * C::kOStride + c1] = o[nd][3];
    }
    if (tid4 == 0) {
      mbuf[warp * 16 + gid] = m_r[0];
      mbuf[warp * 16 + gid + 8] = m_r[1];
      lbuf[warp * 16 + gid] = l_r[0];
      lbuf[warp * 16 + gid + 8] = l_r[1];
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * D; idx += C::kThreads) {
    const int r = idx / D, e = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mbuf[w * 16 + r]);
    float* dst = ws + ((static_cast<int64_t>(i) * Hq + kvh * grp + r) * S + s) * (D + 1);
    if (M == -CUDART_INF_F) {
      dst[e] = 0.f;
      if (e == 0) dst[D] = -CUDART_INF_F;
      continue;
    }
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float f = fast_exp2(mbuf[w * 16 + r] - M);
      L += f * lbuf[w * 16 + r];
      acc += f * cbuf[(w * 16 + r) * C::kOStride + e];
    }
    dst[e] = acc / L * v_scale;
    if (e == 0) dst[D] = (M + log2f(L)) * kLn2;
  }
}

template <int D, int STAGES>
static cudaError_t launch_decode_fp8_t(const void* q, const void* cache,
                                       const int32_t* block_table, const int32_t* seq_lens, int N,
                                       int Hq, int Hkv, int bs, int num_blocks, int max_blocks,
                                       float scale, float k_scale, float v_scale, int S, int chunk,
                                       float* ws, int* err, cudaStream_t stream) {
  using C = DecodeFp8Cfg<D, STAGES>;
  auto kern = decode_splitkv_fp8_kernel<D, STAGES>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(S, Hkv, N), dim3(C::kThreads), C::kSmemBytes, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const uint8_t*>(cache),
                    block_table, seq_lens, max_blocks, Hq, Hkv, bs, num_blocks,
                    scale * k_scale * kLog2e, v_scale, S, chunk, ws, err);
}

cudaError_t launch_decode_splitkv_fp8(const void* q, const void* cache,
                                      const int32_t* block_table, const int32_t* seq_lens, int N,
                                      int Hq, int Hkv, int d, int bs, int num_blocks,
                                      int max_blocks, float scale, float k_scale, float v_scale,
                                      int S, int chunk, float* ws, int* err, cudaStream_t stream) {
  if (d == 128)
    return launch_decode_fp8_t<128, 4>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs,
                                       num_blocks, max_blocks, scale, k_scale, v_scale, S, chunk,
                                       ws, err, stream);
  return launch_decode_fp8_t<64, 8>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs, num_blocks,
                                    max_blocks, scale, k_scale, v_scale, S, chunk, ws, err,
                                    stream);
}

}  // namespace pa
