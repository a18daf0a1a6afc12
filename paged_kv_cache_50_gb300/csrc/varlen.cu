// Varlen paged attention (prefill / chunked prefill / mixed batches): step 2
// of the paged-kernel contract ("Attention Backends", section "What 'paged
// attention' requires of a kernel"): each request attends from its queries
// over its first seq_len tokens, fetched block by block through its
// block_table row, with O = softmax(Q K^T * scale + M) V ("Chapter 1:
// attention backends", section 2.1) and the FlashAttention tiling + online
// softmax of section 4.1 (no score matrix is ever written to HBM).
//
// Tensor-core path for sm_103a with warp-level mma.m16n8k16 tiles:
//  * CTA = (tile of 64 packed rows, kv head, request).  A packed row is one
//    (query row, q head of the kv group) pair, row r -> query r / g, head
//    r % g, so the Hq/Hkv heads that share a kv head share every K/V tile
//    loaded into shared memory;
//  * K/V tiles of 64 tokens (four 16-token pieces of cache blocks) are
//    gathered through the block table with 16-byte cp.async into an
//    XOR-swizzled, double-buffered ring; tokens past the end of the visible
//    range are zero-filled, never read;
//  * each of the 4 warps owns 16 packed rows: S = Q K^T, causal mask
//    (bottom-right: query row j of a request with qlen new tokens sits at
//    position seq - qlen + j), online softmax in registers, O += P V;
//  * the CTA stops at the last tile any of its rows can see.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <int D>
struct VarlenCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = 128;
  static constexpr int kBM = 64;   // packed rows per CTA
  static constexpr int kBN = 64;   // tokens per K/V tile
  static constexpr int kRowBytes = D * 2;
  static constexpr int kChunks = D / 8;
  static constexpr int kTileBytes = kBN * kRowBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = 2 * kStageBytes;
};

__device__ __forceinline__ uint32_t vswz(int row, int chunk, int row_bytes) {
  return static_cast<uint32_t>(row * row_bytes + ((chunk ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(128)
varlen_fwd_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ cache,
                  const int32_t* __restrict__ block_table, const int32_t* __restrict__ qsl,
                  const int32_t* __restrict__ seq_lens, int max_blocks, int Hq, int Hkv, int bs,
                  int num_blocks, float scale_log2, int causal, __nv_bfloat16* __restrict__ out,
                  float* __restrict__ lse, int* err) {
  using C = VarlenCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int i = blockIdx.z, kvh = blockIdx.y;
  const int grp = Hq / Hkv;
  const int q0 = qsl[i];
  const int qlen = qsl[i + 1] - q0;
  const int rows_total = qlen * grp;
  const int row0 = blockIdx.x * C::kBM;
  if (row0 >= rows_total) return;
  const int seq = seq_lens[i];
  const int ctx = seq - qlen;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tid4 = lane & 3;

  // This thread's two packed rows.
  int lim[2];            // number of visible tokens of each row
  int64_t qoff[2];       // element offset of the row's q / out vector
  bool valid[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int pr = row0 + warp * 16 + gid + 8 * r;
    valid[r] = pr < rows_total;
    const int qi = valid[r] ? pr / grp : 0;
    const int hh = valid[r] ? pr % grp : 0;
    lim[r] = valid[r] ? (causal ? ctx + qi + 1 : seq) : 0;
    if (lim[r] > seq) lim[r] = seq;
    if (lim[r] < 0) lim[r] = 0;
    qoff[r] = (static_cast<int64_t>(q0 + qi) * Hq + kvh * grp + hh) * D;
  }
  // Tokens any row of this CTA can see.
  const int last_row = min(row0 + C::kBM, rows_total) - 1;
  int kv_end = causal ? ctx + last_row / grp + 1 : seq;
  kv_end = max(0, min(kv_end, seq));
  const int ntiles = (kv_end + C::kBN - 1) / C::kBN;

  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int c0 = kk * 16 + 2 * tid4;
    qf[kk][0] = valid[0] ? *reinterpret_cast<const uint32_t*>(q + qoff[0] + c0) : 0u;
    qf[kk][1] = valid[1] ? *reinterpret_cast<const uint32_t*>(q + qoff[1] + c0) : 0u;
    qf[kk][2] = valid[0] ? *reinterpret_cast<const uint32_t*>(q + qoff[0] + c0 + 8) : 0u;
    qf[kk][3] = valid[1] ? *reinterpret_cast<const uint32_t*>(q + qoff[1] + c0 + 8) : 0u;
  }

  const uint32_t sbase = smem_u32(smem);
  const int64_t row_stride = static_cast<int64_t>(Hkv) * D;
  const int32_t* table = block_table + static_cast<int64_t>(i) * max_blocks;

  auto issue = [&](int kt) {
    const uint32_t kdst = sbase + (kt & 1) * C::kStageBytes;
    const uint32_t vdst = kdst + C::kTileBytes;
#pragma unroll
    for (int k = 0; k < C::kBN * C::kChunks / C::kThreads; ++k) {
      const int c = threadIdx.x + C::kThreads * k;
      const int r = c / C::kChunks, cc = c % C::kChunks;
      const int tok = kt * C::kBN + r;
      int bytes = 0;
      const __nv_bfloat16* ksrc = cache;
      if (tok < kv_end) {
        const int blk = block_at(table, tok / bs, max_blocks);
        if (blk >= 0 && blk < num_blocks) {
          bytes = 16;
          ksrc = cache + ((static_cast<int64_t>(blk) * 2) * bs + tok % bs) * row_stride +
                 static_cast<int64_t>(kvh) * D + cc * 8;
        } else if (cc == 0) {
          record_error(err, PA_DEVERR_BLOCK_ID);
        }
      }
      const uint32_t so = vswz(r, cc, C::kRowBytes);
      cp_async_16(kdst + so, ksrc, bytes);
      cp_async_16(vdst + so, bytes ? ksrc + static_cast<int64_t>(bs) * row_stride : cache, bytes);
    }
  };

  float m_r[2] = {-CUDART_INF_F, -CUDART_INF_F};
  float l_r[2] = {0.f, 0.f};
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;

  if (ntiles > 0) issue(0);
  cp_async_commit();
  for (int kt = 0; kt < ntiles; ++kt) {
    if (kt + 1 < ntiles) issue(kt + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const uint32_t kb = sbase + (kt & 1) * C::kStageBytes;
    const uint32_t vb = kb + C::kTileBytes;
    const int tok0 = kt * C::kBN;

    // Validity of the four 16-token pieces (a bad block id masks its tokens).
    int vmask = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int t = tok0 + p * 16;
      if (t < kv_end) {
        const int blk = block_at(table, t / bs, max_blocks);
        if (blk >= 0 && blk < num_blocks) vmask |= 1 << p;
      }
    }

    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int tok = np * 16 + (mi >> 1) * 8 + rr;
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(kb + vswz(tok, 2 * kk + (mi & 1), C::kRowBytes), b0, b1, b2, b3);
          mma_bf16_16816(sc[2 * np], qf[kk], b0, b1);
          mma_bf16_16816(sc[2 * np + 1], qf[kk], b2, b3);
        }
      }
    }

    float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = tok0 + nt * 8 + 2 * tid4 + (e & 1);
        const bool vis = tok < lim[e >> 1] && ((vmask >> (nt >> 1)) & 1);
        const float x = vis ? sc[nt][e] * scale_log2 : -CUDART_INF_F;
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
    for (int nt = 0; nt < 8; ++nt)
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

    {
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        uint32_t pf[4];
        pf[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        pf[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        pf[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pf[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const int tok = kk * 16 + (mi & 1) * 8 + rr;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4_trans(vb + vswz(tok, 2 * jj + (mi >> 1), C::kRowBytes), b0, b1, b2, b3);
          mma_bf16_16816(o[2 * jj], pf, b0, b1);
          mma_bf16_16816(o[2 * jj + 1], pf, b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 1);
    l_r[r] += __shfl_xor_sync(0xffffffffu, l_r[r], 2);
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    if (!valid[r]) continue;
    const float inv = l_r[r] > 0.f ? 1.f / l_r[r] : 0.f;
    __nv_bfloat16* dst = out + qoff[r];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      *reinterpret_cast<uint32_t*>(dst + nd * 8 + 2 * tid4) =
          pack_bf16(o[nd][2 * r] * inv, o[nd][2 * r + 1] * inv);
    }
    if (lse != nullptr && tid4 == 0) {
      lse[qoff[r] / D] = l_r[r] > 0.f ? (m_r[r] + log2f(l_r[r])) * kLn2 : -CUDART_INF_F;
    }
  }
}

template <int D>
static cudaError_t launch_varlen_t(const void* q, const void* cache, const int32_t* block_table,
                                   const int32_t* qsl, const int32_t* seq_lens, int N, int Hq,
                                   int Hkv, int bs, int num_blocks, int max_blocks,
                                   int max_query_len, float scale, int causal, void* out,
                                   float* lse, int* err, cudaStream_t stream) {
  using C = VarlenCfg<D>;
  auto kern = varlen_fwd_kernel<D>;
  static DeviceFlags attr_set;
  cudaError_t e = set_smem_once(kern, C::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  const int grp = Hq / Hkv;
  const long long rows = static_cast<long long>(max_query_len) * grp;
  dim3 grid(static_cast<unsigned>((rows + C::kBM - 1) / C::kBM), Hkv, N);
  kern<<<grid, C::kThreads, C::kSmemBytes, stream>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(cache), block_table,
      qsl, seq_lens, max_blocks, Hq, Hkv, bs, num_blocks, scale * kLog2e, causal,
      static_cast<__nv_bfloat16*>(out), lse, err);
  return cudaGetLastError();
}

cudaError_t launch_varlen_fwd(const void* q, const void* cache, const int32_t* block_table,
                              const int32_t* qsl, const int32_t* seq_lens, int N, int Hq, int Hkv,
                              int d, int bs, int num_blocks, int max_blocks, int max_query_len,
                              float scale, int causal, void* out, float* lse,
                              int* err, cudaStream_t stream) {
  if (d == 128)
    return launch_varlen_t<128>(q, cache, block_table, qsl, seq_lens, N, Hq, Hkv, bs, num_blocks,
                                max_blocks, max_query_len, scale, causal, out, lse, err, stream);
  return launch_varlen_t<64>(q, cache, block_table, qsl, seq_lens, N, Hq, Hkv, bs, num_blocks,
                             max_blocks, max_query_len, scale, causal, out, lse, err, stream);
}

}  // namespace pa
