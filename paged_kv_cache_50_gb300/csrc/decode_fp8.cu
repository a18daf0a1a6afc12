// Split-KV decode (stage 1) over an fp8 pool of e4m3 codes,
// [num_blocks, 2, block_size, Hkv, d] bytes.  An entry stands for its e4m3
// value times the layer's k_scale (K half) or v_scale (V half): "Triton and
// MLA" (vllm-arch-zh), data flow -- the decode kernel always receives both
// scales.  The split, the online softmax and the workspace layout
// [N, Hq, S, d + 1] are those of the bf16 stage 1 ("Chapter 1: attention
// backends", sections 3.1 and 4.1); the LSE merge is shared.
//
// GB300 design (HBM-bound in principle; an fp8 pool halves the bytes per
// token, so the instructions spent per token decide whether HBM is reached):
//  * one CTA per (split, kv head, request), four warps taking 16-token
//    sub-blocks round-robin, each warp with its own cp.async ring of raw code
//    tiles (no CTA-wide barrier in the main loop);
//  * the tokens are the M dimension of mma.m16n8k16 and the kv group's query
//    heads its N dimension (8 per n-tile): S^T = K Q^T and O^T += V^T P^T, so
//    a 16-token sub-block costs d/16 MMAs per product and the output state is
//    d/16 x 4 registers per n-tile;
//  * codes go from shared memory straight into operand registers: e4m3 ->
//    f16 is exact (cvt.rn.f16x2.e4m3x2), so the MMAs run on f16 operands, q
//    converted bf16 -> f16 once (exact for |q| in f16's normal range) and the
//    softmax weights packed as f16;
//  * a dot product does not depend on the order of its terms, so the head
//    dimension is permuted alike in K and Q: the 4 k-values a lane owns in
//    k-step kk are the bytes [tid4 * d/4 + 4 kk, + 4) of its token rows, one
//    32-bit word of codes per row;
//  * rows of the V^T operand are permuted too: row gid (gid + 8) of d-tile md
//    is head dimension gid * d/8 + 2 md (+ 1), so a lane's V bytes are d/8
//    contiguous codes of each of its four token rows, paired across rows with
//    byte permutes; the combine writes the dimensions back in order;
//  * the softmax weights leave the MMA as S^T (lane = token) and enter the
//    next one as P^T (lane = head): four shuffles of f16 pairs per n-tile;
//  * the running max is moved only when a sub-block's max exceeds it by more
//    than 8 (log2 units), so the output rescale is rare; weights then stay
//    below 2^8, well inside f16;
//  * k_scale folds into the exp2 scale and v_scale into the partial output
//    (the LSE does not depend on V).
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <int D, int STAGES, int NT>
struct DecodeFp8Cfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunks = D / 16;             // 16-byte chunks per row
  static constexpr int kTileBytes = 16 * D;          // 16 tokens of K (or V) codes
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kWarpBytes = STAGES * kStageBytes;
  static constexpr int kPipeBytes = kWarps * kWarpBytes;
  // Combine buffer: per warp 8*NT head rows of d floats, one pad float after
  // every 16, rows kOStride apart (kOStride = 4 mod 32 keeps the fragment
  // stores free of bank conflicts for d = 128).
  static constexpr int kOStride = D == 128 ? 164 : 68;
  static constexpr int kHeads = 8 * NT;
  static constexpr int kCombineBytes = kWarps * (kHeads * kOStride + 2 * kHeads) * 4;
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

// The lane's `words` 32-bit words of a code row starting at byte `byte0`
// (a multiple of 16 for 16-byte reads, of 8 for 8-byte ones).
template <int D, int WORDS>
__device__ __forceinline__ void load_row_words(uint32_t tile, int r, int byte0,
                                               uint32_t (&w)[WORDS]) {
  if constexpr (WORDS % 4 == 0) {
#pragma unroll
    for (int k = 0; k < WORDS / 4; ++k) {
      const uint4 x = lds128(tile + swz8<D>(r, byte0 / 16 + k));
      w[4 * k] = x.x;
      w[4 * k + 1] = x.y;
      w[4 * k + 2] = x.z;
      w[4 * k + 3] = x.w;
    }
  } else {
    static_assert(WORDS == 2, "8-byte rows only");
    const uint2 x = lds64(tile + swz8<D>(r, byte0 / 16) + (byte0 & 8));
    w[0] = x.x;
    w[1] = x.y;
  }
}

template <int D, int STAGES, int NT>
__global__ void __launch_bounds__(128)
decode_splitkv_fp8_kernel(const __nv_bfloat16* __restrict__ q, const uint8_t* __restrict__ cache,
                          const int32_t* __restrict__ block_table,
                          const int32_t* __restrict__ seq_lens, int max_blocks, int Hq, int Hkv,
                          int bs, int bs_log2, int num_blocks, float scale_log2, float v_scale,
                          int S,
                          int chunk, float* __restrict__ ws, int* err) {
  using C = DecodeFp8Cfg<D, STAGES, NT>;
  constexpr int kK = D / 16;   // k-steps of Q K^T = d-tiles of V^T P^T
  constexpr int kW = D / 32;   // words of V codes per lane per token row
  constexpr float kRescale = 8.f;
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, kvh = blockIdx.y, i = blockIdx.z;
  const int grp = Hq / Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;

  pdl_wait();
  const long long a0 = static_cast<long long>(s) * chunk;
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks;
  // Block ids of the warp's first STAGES sub-blocks, read together with
  // seq_len (they do not depend on it when the split is not empty, which
  // then starts at a0); ids of sub-blocks the split does not have are never
  // used.
  int first_blk[STAGES];
#pragma unroll
  for (int n = 0; n < STAGES; ++n) {
    const long long col = bs_log2 >= 0 ? (a0 + (warp + n * C::kWarps) * 16) >> bs_log2
                                       : (a0 + (warp + n * C::kWarps) * 16) / bs;
    first_blk[n] = col < max_blocks ? block_at(table, static_cast<int>(col), max_blocks) : -1;
  }
  const int seq = seq_lens[i];
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
      ws[((static_cast<int64_t>(i) * Hq + kvh * grp + r) * S + s) * (D + 1) + e] =
          e == D ? -CUDART_INF_F : 0.f;
    }
    return;
  }
  const int my_n = nsb > warp ? (nsb - warp + C::kWarps - 1) / C::kWarps : 0;

  // Q^T as the B operand: lane (gid, tid4) holds head nt*8 + gid (zero past
  // the group), k-values in the permuted order described above.
  uint32_t qf[NT][kK][2];
  {
    const __nv_bfloat16* qb = q + (static_cast<int64_t>(i) * Hq + static_cast<int64_t>(kvh) * grp) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + gid;
      const bool ok = h < grp;
#pragma unroll
      for (int kk = 0; kk < kK; ++kk) {
        const int c0 = tid4 * (D / 4) + kk * 4;
        qf[nt][kk][0] = ok ? q_pair_f16(qb + h * D + c0) : 0u;
        qf[nt][kk][1] = ok ? q_pair_f16(qb + h * D + c0 + 2) : 0u;
      }
    }
  }

  const uint32_t wbase = smem_u32(smem) + warp * C::kWarpBytes;
  const int64_t row_stride = static_cast<int64_t>(Hkv) * D;  // bytes per token row

  // Block id of the warp's n-th sub-block (loaded one iteration before its
  // copies are issued, so the table read is off the critical path).
  auto lookup = [&](int n) {
    return block_at(table, div_bs(t0 + (warp + n * C::kWarps) * 16, bs, bs_log2), max_blocks);
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

  // Per lane: heads nt*8 + 2 tid4 + j (j = 0, 1) -- running max (replicated
  // over the 8 token lanes), partial sums over the lane's tokens, and O^T.
  float m_r[NT][2], l_r[NT][2];
  float o[NT][kK][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_r[nt][0] = m_r[nt][1] = -CUDART_INF_F;
    l_r[nt][0] = l_r[nt][1] = 0.f;
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
      uint32_t k0[D / 16], k1[D / 16];
      load_row_words<D, D / 16>(kb, gid, tid4 * (D / 4), k0);
      load_row_words<D, D / 16>(kb, gid + 8, tid4 * (D / 4), k1);
#pragma unroll
      for (int kk = 0; kk < kK; ++kk) {
        uint32_t a[4];
        e4m3x4_to_f16(k0[kk], a[0], a[2]);
        e4m3x4_to_f16(k1[kk], a[1], a[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_f16_16816(s2[nt][kk & 1], a, qf[nt][kk][0], qf[nt][kk][1]);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] = s2[nt][0][e] + s2[nt][1][e];
    }

    // Online softmax (log2 domain, scale * k_scale folded in), per head over
    // the 16 tokens: two in the lane, the rest across the 8 token lanes.
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
          // Move the reference max (first finite max, or growth past the
          // margin); rescale what was accumulated against the old one.
          const float alpha = fast_exp2(m_r[nt][j] - mx);   // 0 when m_r = -inf
          m_r[nt][j] = mx;
          l_r[nt][j] *= alpha;
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
      // S^T -> P^T: this lane's (token, head pair) values as f16 pairs, then
      // each lane gathers its head's four tokens.
      const uint32_t u_lo = pack_f16(p[0], p[1]);   // token gid, heads 2 tid4, +1
      const uint32_t u_hi = pack_f16(p[2], p[3]);   // token gid + 8
      const uint32_t xa = __shfl_sync(0xffffffffu, u_lo, srcA);
      const uint32_t xb = __shfl_sync(0xffffffffu, u_lo, srcB);
      const uint32_t ya = __shfl_sync(0xffffffffu, u_hi, srcA);
      const uint32_t yb = __shfl_sync(0xffffffffu, u_hi, srcB);
      pb[nt][0] = __byte_perm(xa, xb, psel);
      pb[nt][1] = __byte_perm(ya, yb, psel);
    }

    // O^T += V^T P^T.  The lane's A operand: head dimensions gid * d/8 + c
    // (c < d/8) of tokens 2 tid4 + {0, 1} (rows of a0/a1) and + {8, 9} (a2/a3).
    {
      uint32_t va[kW], vb1[kW], vc[kW], ve[kW];
      const int rA = 2 * tid4, byte0 = gid * (D / 8);
      load_row_words<D, kW>(vb, rA, byte0, va);
      load_row_words<D, kW>(vb, rA + 1, byte0, vb1);
      load_row_words<D, kW>(vb, rA + 8, byte0, vc);
      load_row_words<D, kW>(vb, rA + 9, byte0, ve);
#pragma unroll
      for (int w = 0; w < kW; ++w) {
        // c01[k]: f16 pairs (token 2 tid4, 2 tid4 + 1) of dimension 4w + k;
        // c89[k]: the same for tokens 2 tid4 + 8, + 9.
        uint32_t c01[4], c89[4];
        e4m3x4_to_f16(__byte_perm(va[w], vb1[w], 0x5140), c01[0], c01[1]);
        e4m3x4_to_f16(__byte_perm(va[w], vb1[w], 0x7362), c01[2], c01[3]);
        e4m3x4_to_f16(__byte_perm(vc[w], ve[w], 0x5140), c89[0], c89[1]);
        e4m3x4_to_f16(__byte_perm(vc[w], ve[w], 0x7362), c89[2], c89[3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // d-tile md = 2w + h: row gid = dimension 4w + 2h, row gid + 8 = 4w + 2h + 1.
          const uint32_t a[4] = {c01[2 * h], c01[2 * h + 1], c89[2 * h], c89[2 * h + 1]};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16_16816(o[nt][2 * w + h], a, pb[nt][0], pb[nt][1]);
        }
      }
    }
  }
  cp_async_wait<0>();
  pdl_trigger();

  // Partial sums over the 8 token lanes.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 4);
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 8);
      l_r[nt][j] += __shfl_xor_sync(0xffffffffu, l_r[nt][j], 16);
    }

  // Merge the four warps' states through shared memory: per warp kHeads rows
  // of d floats (dimension e at e + e/16), then max and sum per head.
  __syncthreads();
  float* cbuf = reinterpret_cast<float*>(smem);
  float* mbuf = cbuf + C::kWarps * C::kHeads * C::kOStride;  // [warp][kHeads]
  float* lbuf = mbuf + C::kWarps * C::kHeads;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int md = 0; md < kK; ++md) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int h = nt * 8 + 2 * tid4 + (e & 1);
        const int dim = gid * (D / 8) + 2 * md + (e >> 1);
        cbuf[(warp * C::kHeads + h) * C::kOStride + dim + (dim >> 4)] = o[nt][md][e];
      }
    }
    if (gid == 0) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        mbuf[warp * C::kHeads + nt * 8 + 2 * tid4 + j] = m_r[nt][j];
        lbuf[warp * C::kHeads + nt * 8 + 2 * tid4 + j] = l_r[nt][j];
      }
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < grp * D; idx += C::kThreads) {
    const int r = idx / D, e = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) M = fmaxf(M, mbuf[w * C::kHeads + r]);
    float* dst = ws + ((static_cast<int64_t>(i) * Hq + kvh * grp + r) * S + s) * (D + 1);
    if (M == -CUDART_INF_F) {
      dst[e] = 0.f;
      if (e == 0) dst[D] = -CUDART_INF_F;
      continue;
    }
    float L = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float f = fast_exp2(mbuf[w * C::kHeads + r] - M);
      L += f * lbuf[w * C::kHeads + r];
      acc += f * cbuf[(w * C::kHeads + r) * C::kOStride + e + (e >> 4)];
    }
    dst[e] = acc / L * v_scale;
    if (e == 0) dst[D] = (M + log2f(L)) * kLn2;
  }
}

template <int D, int STAGES, int NT>
static cudaError_t launch_decode_fp8_t(const void* q, const void* cache,
                                       const int32_t* block_table, const int32_t* seq_lens, int N,
                                       int Hq, int Hkv, int bs, int num_blocks, int max_blocks,
                                       float scale, float k_scale, float v_scale, int S, int chunk,
                                       float* ws, int* err, cudaStream_t stream) {
  using C = DecodeFp8Cfg<D, STAGES, NT>;
  auto kern = decode_splitkv_fp8_kernel<D, STAGES, NT>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(S, Hkv, N), dim3(C::kThreads), C::kSmemBytes, stream,
                    static_cast<const __nv_bfloat16*>(q), static_cast<const uint8_t*>(cache),
                    block_table, seq_lens, max_blocks, Hq, Hkv, bs, block_size_log2(bs), num_blocks,
                    scale * k_scale * kLog2e, v_scale, S, chunk, ws, err);
}

cudaError_t launch_decode_splitkv_fp8(const void* q, const void* cache,
                                      const int32_t* block_table, const int32_t* seq_lens, int N,
                                      int Hq, int Hkv, int d, int bs, int num_blocks,
                                      int max_blocks, float scale, float k_scale, float v_scale,
                                      int S, int chunk, float* ws, int* err, cudaStream_t stream) {
  const bool wide = Hq / Hkv > 8;   // groups of 9..16 heads take two n-tiles
#define PA_FP8_LAUNCH(DD, ST, NTT)                                                              \
  return launch_decode_fp8_t<DD, ST, NTT>(q, cache, block_table, seq_lens, N, Hq, Hkv, bs,      \
                                          num_blocks, max_blocks, scale, k_scale, v_scale, S,   \
                                          chunk, ws, err, stream)
  if (d == 128) {
    if (wide) PA_FP8_LAUNCH(128, 4, 2);
    PA_FP8_LAUNCH(128, 3, 1);
  }
  if (wide) PA_FP8_LAUNCH(64, 8, 2);
  PA_FP8_LAUNCH(64, 8, 1);
#undef PA_FP8_LAUNCH
}

}  // namespace pa
