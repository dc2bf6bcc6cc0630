// Causal varlen GQA prefill attention on GB300 tensor cores: tcgen05 MMAs
// with TMEM accumulators, K/V tiles moved by TMA ([SK] §7.2, flash-attention
// style online softmax).
//
// One CTA owns two "units" of 128 query rows that read the same kv head:
// two q heads of one GQA group at the same query tile when the group size is
// even, else two consecutive query tiles of one head.  Per CTA (10 warps):
//   warp 0      TMA producer: K_j and V_j tiles (128 keys x 128 dims, two
//               128-byte-swizzled boxes of 64 dims), two slots each
//   warp 1      allocates 512 TMEM columns and issues every MMA from one
//               thread:
//                 S_u  = Q_u K_j^T   A = Q_u (smem), B = K_j (smem), both K-major
//                 O_u += P_u V_j     A = P_u (TMEM), B = V_j (smem, MN-major)
//               in the order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): one unit's
//               softmax runs while the tensor pipe works on the other's MMAs.
//               The issuing thread waits on as few barriers as possible
//               (barrier operations are slow while the MMAs saturate shared
//               memory): a unit's P-ready signal also certifies that V_j and
//               K_{j+1} have landed, which its softmax warps checked.
//   warps 2-5   softmax of unit 0, warps 6-9 of unit 1: one query row per
//               thread (TMEM lane = row).  S is read with tcgen05.ld, masked,
//               the online max / sum kept in fp32, and P = exp2(...) rounded
//               to bf16 is written back with tcgen05.st over the first 64
//               columns of the same S buffer (two bf16 per column), where
//               the PV MMA reads it.  S_u(j+1) is issued only after PV_u(j)
//               has completed, so it never overwrites a P still in use.
// TMEM columns: S_0/P_0 [0,128), S_1/P_1 [128,256), O_0 [256,384), O_1 [384,512).
// The running max is raised lazily: O and l are rescaled only when a row's
// max grows by more than 2^8, which keeps every P <= 256 and is exact because
// O and l always share the same reference max.  The final O / l is staged in
// shared memory and stored coalesced.
// Every mbarrier wait is bounded (2 s); on timeout the kernel records an
// error word and runs to completion without waiting further.
#include <math.h>

#include "common.cuh"
#include "tc_common.cuh"

namespace qw {
namespace pfa {

__device__ unsigned int g_prefill_timeout = 0;

constexpr int HD = 128;        // head_dim
constexpr int BM = 128;        // query rows per unit (MMA M)
constexpr int BN = 128;        // keys per tile
constexpr int THREADS = 320;
constexpr uint32_t BOX = 16384;                     // 128 rows x 64 bf16
constexpr uint32_t TILE = 2 * BOX;                  // 128 rows x 128 bf16
constexpr uint32_t OFF_Q = 0;                       // Q_0, Q_1 (then the output staging)
constexpr uint32_t OFF_K = 2 * TILE;                // K_j in slot j % 2
constexpr uint32_t OFF_V = 4 * TILE;                // V_j in slot j % 2
constexpr uint32_t OFF_BAR = 6 * TILE;
constexpr size_t SMEM = 1024 + OFF_BAR + 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleLog2 = 8.0f;

// barrier indices
constexpr int B_K_FULL = 0, B_K_EMPTY = 2, B_V_FULL = 4, B_V_EMPTY = 6, B_Q = 8, B_S_FULL = 10, B_P_FULL = 12,
              B_O_DONE = 14, B_VTAIL = 16, B_DONE = 17, N_BARS = 18;
static_assert(N_BARS * 8 + 4 <= 256, "barrier area");

constexpr uint32_t IDESC_S = tcx::idesc_bf16(BM, BN);
constexpr uint32_t IDESC_PV = tcx::idesc_bf16(BM, HD) | tcx::kIdescBMajorMN;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// byte offset of (row r, 16-byte chunk c of 16) in a [128][128] bf16 tile
// stored as two 128-byte-swizzled boxes of 64 columns
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return uint32_t(c >> 3) * BOX + uint32_t(r) * 128u + (uint32_t((c & 7) ^ (r & 7)) << 4);
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T (A: lane = row, two bf16 per 32-bit column)
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(THREADS, 1) attn_prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const bf16* __restrict__ q,
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, const int32_t* __restrict__ seq_base,
    int nh, int nkv, int pair_heads, float scale_log2, bf16* __restrict__ out, const KvPages pages) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(sm);
  const uint32_t bar0 = sbase + OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * uint32_t(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_BAR + N_BARS * 8);

  const int s = blockIdx.z;
  const int qs = cu_q[s];
  const int Lq = cu_q[s + 1] - qs;
  const int Lk = cu_k[s + 1] - cu_k[s];
  const int offset = Lk - Lq;
  const int qt = int(gridDim.x) - 1 - int(blockIdx.x);   // longest (causal) tiles first
  int h_u[2], qlo[2], n_u[2];
  if (pair_heads) {
    h_u[0] = 2 * int(blockIdx.y);
    h_u[1] = h_u[0] + 1;
    qlo[0] = qlo[1] = qt * BM;
  } else {
    h_u[0] = h_u[1] = int(blockIdx.y);
    qlo[0] = qt * 2 * BM;
    qlo[1] = qlo[0] + BM;
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int kv_end = qlo[u] < Lq ? min(Lk, offset + min(Lq, qlo[u] + BM)) : 0;
    n_u[u] = (kv_end + BN - 1) / BN;
  }
  const int n_kv = max(n_u[0], n_u[1]);
  if (n_kv == 0) return;   // uniform over the CTA, before any barrier or TMEM use
  const int g = h_u[0] / (nh / nkv);
  const int64_t kbase = seq_base != nullptr ? int64_t(seq_base[s]) : int64_t(cu_k[s]);
  const int warp = int(threadIdx.x) >> 5, lane = int(threadIdx.x) & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      tcx::mbar_init(bar(B_K_FULL + i), 1);
      tcx::mbar_init(bar(B_K_EMPTY + i), 1);
      tcx::mbar_init(bar(B_V_FULL + i), 1);
      tcx::mbar_init(bar(B_V_EMPTY + i), 1);
      tcx::mbar_init(bar(B_Q + i), BM);
      tcx::mbar_init(bar(B_S_FULL + i), 1);
      tcx::mbar_init(bar(B_P_FULL + i), 4);
      tcx::mbar_init(bar(B_O_DONE + i), 1);
    }
    tcx::mbar_init(bar(B_VTAIL), 1);
    tcx::mbar_init(bar(B_DONE), 1);
    tcx::fence_mbar_init();
    tcx::prefetch_map(&tmK);
    tcx::prefetch_map(&tmV);
  }
  if (warp == 1) {
    tcx::tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tcx::tmem_relinquish();
  }
  tcx::tc_fence_before();
  __syncthreads();
  tcx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  auto wait = [&](int b, uint32_t parity, uint32_t code) {
    if (ok && !tcx::mbar_wait(bar(b), parity, &g_prefill_timeout, 1u << code)) ok = false;
  };

  if (warp == 0) {
    // ---------------- TMA producer: K_0, then K_{j+1}, V_j for j = 0, 1, ... ----------------
    auto load = [&](uint32_t dst, const CUtensorMap* map, uint32_t b, int j) {
      if (lane == 0) {
        tcx::mbar_expect_tx(b, TILE);
        // cache row of key j * BN: contiguous from kbase, or through the block table
        const int row = pages.table == nullptr ? int(kbase) + j * BN
                                               : pages.table[int64_t(s) * pages.max_blocks + j * BN / pages.block_size] *
                                                         pages.block_size +
                                                     (j * BN) % pages.block_size;
        tcx::tma_load_3d(dst, map, b, 0, g, row);
        tcx::tma_load_3d(dst + BOX, map, b, 64, g, row);
      }
    };
    auto load_k = [&](int j) {
      const int slot = j & 1;
      if (j >= 2) wait(B_K_EMPTY + slot, uint32_t((j >> 1) - 1) & 1u, 1u);
      load(sbase + OFF_K + uint32_t(slot) * TILE, &tmK, bar(B_K_FULL + slot), j);
    };
    load_k(0);
    for (int j = 0; j < n_kv; ++j) {
      if (j + 1 < n_kv) load_k(j + 1);
      const int slot = j & 1;
      if (j >= 2) wait(B_V_EMPTY + slot, uint32_t((j >> 1) - 1) & 1u, 2u);
      const bool tail = j * BN + BN > Lk;   // keys >= Lk in this V tile: zero them
      load(sbase + OFF_V + uint32_t(slot) * TILE, &tmV, bar(tail ? B_VTAIL : B_V_FULL + slot), j);
      if (tail) {
        // whatever the rows past the sequence hold, P is 0 there and 0 * V must stay 0
        wait(B_VTAIL, 0u, 3u);
        const int r0 = Lk - j * BN;
        for (int idx = r0 * 16 + lane; idx < BN * 16; idx += 32)
          *reinterpret_cast<uint4*>(sm + OFF_V + slot * TILE + tile_off(idx >> 4, idx & 15)) =
              make_uint4(0u, 0u, 0u, 0u);
        tcx::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tcx::mbar_arrive(bar(B_V_FULL + slot));
      }
      __syncwarp();
    }
    // drain: the last loads have landed before this CTA may exit
    for (int j = max(0, n_kv - 2); j < n_kv; ++j) {
      wait(B_K_FULL + (j & 1), uint32_t(j >> 1) & 1u, 4u);
      wait(B_V_FULL + (j & 1), uint32_t(j >> 1) & 1u, 4u);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread) ----------------
    if (lane == 0) {
      auto issue_s = [&](int u, int j) {   // S_u(j) = Q_u K_j^T
        const uint32_t qaddr = sbase + OFF_Q + uint32_t(u) * TILE;
        const uint32_t kaddr = sbase + OFF_K + uint32_t(j & 1) * TILE;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = uint32_t(kk >> 2) * BOX + uint32_t(kk & 3) * 32u;
          tcx::umma_bf16(tmem + uint32_t(u) * 128u, tcx::sw128_desc(qaddr + off), tcx::sw128_desc(kaddr + off),
                         IDESC_S, kk > 0 ? 1u : 0u);
        }
        tcx::umma_commit(bar(B_S_FULL + u));
      };
      auto issue_pv = [&](int u, int j) {   // O_u += P_u V_j
        const uint32_t vaddr = sbase + OFF_V + uint32_t(j & 1) * TILE;
        const uint32_t tS = tmem + uint32_t(u) * 128u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_bf16_ts(tS + 256u, tS + uint32_t(kk) * 8u, tcx::sw128_desc_mn(vaddr + uint32_t(kk) * 2048u, BOX),
                       IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        tcx::umma_commit(bar(B_O_DONE + u));
      };
      if (n_u[0] > 0) wait(B_Q, 0u, 5u);
      if (n_u[1] > 0) wait(B_Q + 1, 0u, 5u);
      wait(B_K_FULL, 0u, 6u);
      tcx::tc_fence_after();
      if (n_u[0] > 0) issue_s(0, 0);
      if (n_u[1] > 0) issue_s(1, 0);
      tcx::umma_commit(bar(B_K_EMPTY));   // K_0 released once both S(0) complete
      for (int j = 0; j < n_kv; ++j) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (j < n_u[u]) {
            // P_u(j) written; its softmax also saw V_j (and K_{j+1}) land
            wait(B_P_FULL + u, uint32_t(j) & 1u, 8u);
            tcx::tc_fence_after();
            issue_pv(u, j);
            if (j + 1 < n_u[u]) {
              // S_u(j+1) overwrites the P_u(j) that PV_u(j) reads
              wait(B_O_DONE + u, uint32_t(j) & 1u, 10u);
              tcx::tc_fence_after();
              issue_s(u, j + 1);
            }
          }
        }
        tcx::umma_commit(bar(B_V_EMPTY + (j & 1)));
        if (j + 1 < n_kv) tcx::umma_commit(bar(B_K_EMPTY + ((j + 1) & 1)));
      }
      // every MMA of this CTA has completed before TMEM is released
      tcx::umma_commit(bar(B_DONE));
      wait(B_DONE, 0u, 11u);
    }
    __syncwarp();
  } else {
    // ---------------- softmax (one query row per thread) ----------------
    const int u = (warp - 2) >> 2;            // warps 2-9
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;        // query row within the unit
    const int t128 = (warp - 2 - 4 * u) * 32 + lane;
    const int nu = u ? n_u[1] : n_u[0];
    const int qlo_u = u ? qlo[1] : qlo[0];
    const int head = u ? h_u[1] : h_u[0];
    const int64_t row_stride = int64_t(nh) * HD;
    uint8_t* sQ = sm + OFF_Q + u * TILE;
    if (nu > 0) {
      const bool valid = qlo_u + r < Lq;
      const bf16* src = q + (int64_t(qs) + (valid ? qlo_u + r : 0)) * row_stride + int64_t(head) * HD;
#pragma unroll
      for (int c = 0; c < 16; ++c) cp_async16_zfill(smem_u32(sQ) + tile_off(r, c), src + 8 * c, valid);
      cp_async_commit();
      cp_async_wait<0>();
      tcx::fence_proxy_async();
      tcx::mbar_arrive(bar(B_Q + u));

      const int last_key = min(offset + qlo_u + r, Lk - 1);   // last key this row sees
      const uint32_t tS = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(u) * 128u;
      const uint32_t tO = tS + 256u;
      float m = -INFINITY, l = 0.0f;
      for (int j = 0; j < nu; ++j) {
        // S_u(j) complete, and with it every earlier MMA (O_u holds PV_u(j-1))
        wait(B_S_FULL + u, uint32_t(j) & 1u, 12u);
        tcx::tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tcx::tmem_ld32(tS + 32u * c, sr[c]);
        tcx::tmem_ld_wait();
        const int lim = last_key - j * BN;   // columns > lim are masked
        if (lim < BN - 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent chains
#pragma unroll
        for (int e = 0; e < 32; ++e)
#pragma unroll
          for (int c = 0; c < 4; ++c) mq[c] = fmaxf(mq[c], __uint_as_float(sr[c][e]));
        const float m_tile = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * scale_log2;
        float alpha = 1.0f;
        bool rescale = false;
        if (m_tile > m + kRescaleLog2) {
          alpha = ex2(m - m_tile);
          m = m_tile;
          rescale = true;
        }
        const float m_use = m == -INFINITY ? 0.0f : m;
        float sum0 = 0.0f, sum1 = 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int e = 64 * c + 2 * i;
            const float p0 = ex2(fmaf(__uint_as_float(sr[e >> 5][e & 31]), scale_log2, -m_use));
            const float p1 = ex2(fmaf(__uint_as_float(sr[e >> 5][(e & 31) + 1]), scale_log2, -m_use));
            sum0 += p0;
            sum1 += p1;
            pk[i] = pack_bf16(p0, p1);
          }
          tcx::tmem_st32(tS + 32u * c, pk);   // P_u(j): keys 64c .. 64c+63
        }
        l = l * alpha + (sum0 + sum1);
        if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tcx::tmem_ld32(tO + 32u * c, o);
            tcx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tcx::tmem_st32(tO + 32u * c, o);
          }
        }
        tcx::tmem_st_wait();
        // the MMA thread issues PV_u(j) and S_u(j+1) on this signal alone
        wait(B_V_FULL + (j & 1), uint32_t(j >> 1) & 1u, 14u);
        if (j + 1 < nu) wait(B_K_FULL + ((j + 1) & 1), uint32_t((j + 1) >> 1) & 1u, 14u);
        tcx::tc_fence_before();
        __syncwarp();
        if (lane == 0) tcx::mbar_arrive(bar(B_P_FULL + u));
      }
      // epilogue: O / l -> bf16, staged in Q_u (every S_u MMA completed before the last PV_u),
      // stored coalesced
      wait(B_O_DONE + u, uint32_t(nu - 1) & 1u, 13u);
      tcx::tc_fence_after();
      uint8_t* sO = sQ;
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tcx::tmem_ld32(tO + 32u * c, o);
        tcx::tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(sO + tile_off(r, 4 * c + k)) =
              make_uint4(pack_bf16(__uint_as_float(o[8 * k]) * inv, __uint_as_float(o[8 * k + 1]) * inv),
                         pack_bf16(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv),
                         pack_bf16(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv),
                         pack_bf16(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv));
      }
      tcx::tc_fence_before();
      named_sync(1 + u, 128);
      const int cc = t128 & 15;
#pragma unroll 4
      for (int it = 0; it < BM / 8; ++it) {
        const int rr = it * 8 + (t128 >> 4);
        if (qlo_u + rr < Lq)
          *reinterpret_cast<uint4*>(out + (int64_t(qs) + qlo_u + rr) * row_stride + int64_t(head) * HD + 8 * cc) =
              *reinterpret_cast<const uint4*>(sO + tile_off(rr, cc));
      }
    }
  }
  tcx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tcx::tc_fence_after();
    tcx::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace pfa

unsigned int take_prefill_timeouts() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, pfa::g_prefill_timeout, sizeof(v));
  if (v) cudaMemcpyToSymbol(pfa::g_prefill_timeout, &z, sizeof(z));
  return v;
}

// bf16, head_dim 128: k and v hold kv_rows rows of [nkv, 128]; argument
// checks are done by the caller (qw_attention_prefill).
int launch_attention_prefill_tc(const void* q, const void* k, const void* v, int64_t kv_rows, const int32_t* cu_q,
                                const int32_t* cu_k, const int32_t* seq_base, int n_seqs, int max_seqlen_q, int nh,
                                int nkv, float scale, void* out, cudaStream_t st, const KvPages& pages) {
  using namespace pfa;
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  CUtensorMap mk, mv;
  const uint64_t dims[3] = {uint64_t(HD), uint64_t(nkv), uint64_t(kv_rows)};
  const uint64_t strides[2] = {uint64_t(HD) * 2, uint64_t(nkv) * HD * 2};
  const uint32_t box[3] = {64u, 1u, uint32_t(BN)};
  int rc = make_tensor_map(&mk, k, 3, dims, strides, box);
  if (rc) return rc;
  rc = make_tensor_map(&mv, v, 3, dims, strides, box);
  if (rc) return rc;
  const int G = nh / nkv;
  const int pair = G % 2 == 0;
  const int rows_per_cta = pair ? BM : 2 * BM;
  dim3 grid(unsigned((max_seqlen_q + rows_per_cta - 1) / rows_per_cta), unsigned(pair ? nh / 2 : nh),
            unsigned(n_seqs));
  constexpr float kLog2e = 1.4426950408889634f;
  launch_pdl(attn_prefill_tc_kernel, grid, THREADS, SMEM, st, mk, mv, static_cast<const bf16*>(q), cu_q, cu_k,
             seq_base, nh, nkv, pair, scale * kLog2e, static_cast<bf16*>(out), pages);
  return check_launch("attn_prefill_tc_kernel");
}

}  // namespace qw
