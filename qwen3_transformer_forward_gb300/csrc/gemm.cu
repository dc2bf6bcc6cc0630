// Linear layers of the Qwen3 forward pass on GB300 tensor cores.
//
// C = A W^T in the tensor-parallel layouts of the parallel Linear family
// ([TP] §3-§4, [SK] §5):
//   COLUMN      W [N, K], tp shards stacked along N (merged QKV, gate_up, lm_head)
//   ROW_REDUCE  W [tp, N, K/tp]; the shard partial sums are accumulated in
//               the same fp32 TMEM accumulator (the emulated all_reduce)
//   SILU_MUL    fused SiluAndMul epilogue on a merged gate_up ([SK] §4)
//
// bf16 path: one CTA of 6 warps per 128 x BN output tile.
//   warp 0      TMA producer: 64-wide K slabs of both operands into a
//               STAGES-deep shared-memory ring (128-byte swizzle)
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=16)
//               from one thread; tcgen05.commit frees ring slots
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, convert,
//               store (or fp32 split-K partials)
// Prefill (many tokens): MMA-A = activations, MMA-B = weights, BN = 256.
// Few tokens (<= 64): operands swapped (MMA-A = 128 weight rows,
// MMA-B = the tokens padded to 16/32/64) and split along K so that enough
// CTAs stream the weights -- when the planner finds one split enough (the
// lm_head's 151936 rows) or K does not suit the warp-level GEMV; otherwise
// the few-token GEMV below (gemv_mma_kernel) runs.  The K-splits of one weight tile form a thread-
// block cluster (<= 8 CTAs): each leaves its fp32 partial tile in its own
// shared memory and cluster rank 0 sums them in split order over distributed
// shared memory, then applies the epilogue (bf16, or SiluAndMul with 64 gate
// + 64 up rows per tile).  No global scratch, deterministic.
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on timeout the kernel
// records an error word, drains its own copies and frees TMEM.
//
// f32 path: exact fp32 FMA on CUDA cores (used by the small fp32 model).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <math.h>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "common.cuh"
#include "tc_common.cuh"

namespace qw {

template <typename T>
int launch_gather_rows(const void* src, int64_t n_src, const int32_t* idx, int64_t n, int64_t H, void* out,
                       cudaStream_t st);
template <typename T>
int launch_argmax(const void* logits, int64_t M, int64_t V, int64_t* out, cudaStream_t st);

namespace tc {

using tcx::idesc_bf16;
using tcx::sw128_desc;
using tcx::tc_fence_after;
using tcx::tc_fence_before;
using tcx::tmem_alloc;
using tcx::tmem_dealloc;
using tcx::tmem_ld32;
using tcx::tmem_ld_wait;
using tcx::tmem_relinquish;
using tcx::umma_bf16;
using tcx::umma_commit;

__device__ unsigned int g_tc_timeout = 0;

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int EPI_NONE = 0, EPI_SILU = 1, EPI_QKV = 2, EPI_ADDNORM = 3;
constexpr int kMaxCluster = 8;   // portable cluster size: K-splits per weight tile

struct TcArgs {
  bf16* C;              // output (bf16)
  int splits;           // K-splits per weight tile (= cluster size along y; 1 = direct store)
  int64_t ldc;          // output row stride
  int64_t M;            // token rows
  int64_t N;            // output features (full width before SiluAndMul)
  int p_tiles, q_tiles; // tiles along MMA-A rows (128) and MMA-B rows (BN)
  int p_fastest;        // raster order
  int kblocks;          // k-blocks per split
  int kblocks_total;
  int kpb;              // k-blocks per shard (ROW_REDUCE)
  int64_t k_shard;      // K / tp
  int64_t i_l;          // intermediate per shard (SILU)
  int silu_tps;         // output tiles per shard (SILU)
  int tma_store;        // persistent kernel: the epilogue stores 32 x 64 boxes through tmC
  // EPI_QKV: per-head QK-RMSNorm + RoPE + KV-cache store on the merged QKV output
  const int64_t* positions;
  const float* cos_sin;  // [max_pos, 128]: cos | sin
  int64_t max_pos;
  const bf16* q_gamma;
  const bf16* k_gamma;
  float eps;
  const int64_t* slots;  // cache row per token, -1 = not stored
  bf16* k_cache;
  bf16* v_cache;
  int64_t num_slots;
  bf16* q_out;           // [M, nh, 128]
  int32_t* err;
  int nh, nkv, tp;
  // EPI_ADDNORM: resid <- round(round(C) + resid); y = RMSNorm(resid) * norm_gamma (the
  // row's N columns span the cluster's CTAs; eps as above)
  bf16* resid;
  bf16* y_out;
  const bf16* norm_gamma;
};

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase of parity `parity`; gives up after kTimeoutNs, recording `code`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicOr(&g_tc_timeout, code);
      return false;
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// shared -> global tensor copy of one box (bulk async-group completion)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// at most one of this thread's bulk groups still reading its shared memory source
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every bulk group of this thread complete (its writes performed)
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ float silu_mul_bf16(float g, float u) {
  // gate_up is a model-dtype tensor before SiluAndMul: round both halves first.
  // The fast exp and divide intrinsics (a few fp32 ulp) sit far below the bf16
  // rounding of the result; the accurate ones kept the prefill gate_up
  // epilogue on the transcendental pipe.  (For g -> -inf: 1 + e -> inf and
  // the quotient -> 0, as SiLU.)
  g = round_t<bf16>(g);
  u = round_t<bf16>(u);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// Epilogue tensor stores.  An epilogue warp owns 32 accumulator rows (TMEM
// lanes); it converts 32 rows x 64 columns at a time into one of its two
// staging boxes in shared memory (row r at 128 r bytes, 16-byte chunk v at
// (v ^ (r & 7)) * 16: the 128-byte swizzle of the output tensor map) and
// stores the box with one tensor copy, which clips rows and columns past the
// tensor.  The copies write whole lines and leave the load/store path free;
// direct stores of one row per thread touch 32 rows per instruction.
constexpr uint32_t P_STAGE_BOX = 32 * 128;   // one staging box
struct BoxStore {
  uint32_t stage;   // this warp's two boxes (1024-byte aligned)
  int lane;
  int n = 0;        // boxes stored
  __device__ uint32_t next() {   // a box whose previous copy has read it
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
    return stage + uint32_t(n & 1) * P_STAGE_BOX;
  }
  __device__ void put(uint32_t box, int v, uint4 u) const {
    st_shared_v4(box + uint32_t(lane) * 128u + (uint32_t(v ^ (lane & 7)) << 4), u);
  }
  __device__ void store(const CUtensorMap* map, uint32_t box, int64_t x, int64_t y) {
    tcx::fence_proxy_async();   // the warp's generic writes before the tensor copy reads them
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, box, int(x), int(y));
      bulk_commit();
    }
    ++n;
  }
  __device__ void finish() const {   // the copies have written global memory
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
};
__device__ __forceinline__ uint4 pack8(const uint32_t* q) {
  uint4 u;
  u.x = pack_bf16(__uint_as_float(q[0]), __uint_as_float(q[1]));
  u.y = pack_bf16(__uint_as_float(q[2]), __uint_as_float(q[3]));
  u.z = pack_bf16(__uint_as_float(q[4]), __uint_as_float(q[5]));
  u.w = pack_bf16(__uint_as_float(q[6]), __uint_as_float(q[7]));
  return u;
}
// C[m0 .. m0+31, n_base .. n_base+ncols) = the warp's accumulator columns [0, ncols), as bf16
// (zero: store zeros instead, for a tile with no k-blocks or after a timeout)
__device__ __forceinline__ void epi_store_tma(BoxStore& bs, const CUtensorMap* map, uint32_t trow, int ncols,
                                              int64_t m0, int64_t M, int64_t n_base, int64_t N, bool zero) {
#pragma unroll 1
  for (int c = 0; c < ncols; c += 64) {
    uint32_t r0[32], r1[32];
    tmem_ld32(trow + c, r0);
    tmem_ld32(trow + c + 32, r1);
    tmem_ld_wait();
    if (m0 >= M || n_base + c >= N) continue;   // (warp-uniform)
    if (zero) {
#pragma unroll
      for (int e = 0; e < 32; ++e) r0[e] = r1[e] = 0u;
    }
    const uint32_t box = bs.next();
#pragma unroll
    for (int v = 0; v < 8; ++v) bs.put(box, v, pack8(v < 4 ? r0 + 8 * v : r1 + 8 * (v - 4)));
    bs.store(map, box, n_base + c, m0);
  }
}
// SiluAndMul: gate columns [0, half), up columns [half, 2 half) of the warp's
// accumulator rows -> C[m0 .., col_base + j) for j < half with jl0 + j < i_l
// (i_l % 64 == 0, so that a box never crosses into the next shard's columns)
__device__ __forceinline__ void epi_silu_tma(BoxStore& bs, const CUtensorMap* map, uint32_t trow, int half,
                                             int64_t m0, int64_t M, int64_t col_base, int64_t jl0, int64_t i_l,
                                             bool zero) {
#pragma unroll 1
  for (int c = 0; c < half; c += 64) {
    const bool live = m0 < M && jl0 + c < i_l;   // (warp-uniform)
    const uint32_t box = live ? bs.next() : 0u;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      uint32_t g[32], u[32];
      tmem_ld32(trow + c + 32 * h, g);
      tmem_ld32(trow + half + c + 32 * h, u);
      tmem_ld_wait();
      if (!live) continue;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          o[e] = zero ? 0.0f : silu_mul_bf16(__uint_as_float(g[8 * v + e]), __uint_as_float(u[8 * v + e]));
        uint4 w;
        w.x = pack_bf16(o[0], o[1]);
        w.y = pack_bf16(o[2], o[3]);
        w.z = pack_bf16(o[4], o[5]);
        w.w = pack_bf16(o[6], o[7]);
        bs.put(box, 4 * h + v, w);
      }
    }
    if (live) bs.store(map, box, col_base + c, m0);
  }
}

// Direct stores, one row per thread: row m of the warp's accumulator columns
// [0, ncols) -> C[m, n_base + c] for n_base + c < N (zero: zeros instead)
__device__ __forceinline__ void epi_store_direct(uint32_t trow, int ncols, int64_t m, const TcArgs& a, int64_t n_base,
                                                 bool zero) {
#pragma unroll 1
  for (int c = 0; c < ncols; c += 32) {
    uint32_t r[32];
    tmem_ld32(trow + c, r);
    tmem_ld_wait();
    if (zero) {
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = 0u;
    }
    const int64_t n0 = n_base + c;
    if (m < a.M) {
      bf16* dst = a.C + m * a.ldc + n0;
      if (n0 + 32 <= a.N) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int v = 0; v < 4; ++v) d4[v] = pack8(r + 8 * v);
      } else {
        for (int e = 0; e < 32; ++e)
          if (n0 + e < a.N) dst[e] = __float2bfloat16_rn(__uint_as_float(r[e]));
      }
    }
  }
}
// SiluAndMul, direct stores: gate columns [0, half), up [half, 2 half) of row m
// -> C[m, r_s * i_l + jl0 + j] for jl0 + j < i_l (nothing when !live)
__device__ __forceinline__ void epi_silu_direct(uint32_t trow, int half, int64_t m, const TcArgs& a, int r_s,
                                                int64_t jl0, bool live) {
#pragma unroll 1
  for (int c = 0; c < half; c += 32) {
    uint32_t g[32], u[32];
    tmem_ld32(trow + c, g);
    tmem_ld32(trow + half + c, u);
    tmem_ld_wait();
    if (m < a.M && live) {
      const int64_t j0 = jl0 + c;
      bf16* dst = a.C + m * a.ldc + int64_t(r_s) * a.i_l + j0;
      if (j0 + 32 <= a.i_l) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = silu_mul_bf16(__uint_as_float(g[8 * v + e]), __uint_as_float(u[8 * v + e]));
          uint4 w;
          w.x = pack_bf16(o[0], o[1]);
          w.y = pack_bf16(o[2], o[3]);
          w.z = pack_bf16(o[4], o[5]);
          w.w = pack_bf16(o[6], o[7]);
          d4[v] = w;
        }
      } else {
        for (int e = 0; e < 32; ++e)
          if (j0 + e < a.i_l) dst[e] = __float2bfloat16_rn(silu_mul_bf16(__uint_as_float(g[e]), __uint_as_float(u[e])));
      }
    }
  }
}

// Epilogue of a QKV tile (EPI_QKV): the tile's 256 columns are two whole heads
// of the merged QKV output (shard r = [q_r | k_r | v_r], 128 columns per
// head).  Each thread owns one token row: it rounds the accumulator to the
// bf16 QKV value, then a q or k head is normed, rotated and written (q_out /
// k cache), a v head is copied into the v cache, with the arithmetic of the
// standalone kernel.  trow: this thread's TMEM lane at the tile's column 0.
__device__ __forceinline__ void epi_qkv_tile(const TcArgs& a, uint32_t trow, int64_t m, int tile_q, bool row_ok) {
  constexpr int BN = 256;
  int64_t pos = 0, slot = -1;
  if (m < a.M) {
    pos = a.positions[m];
    slot = a.slots[m];
  }
  const bool pos_ok = pos >= 0 && pos < a.max_pos;
  const int nh_l = a.nh / a.tp, nkv_l = a.nkv / a.tp;
  const int64_t width_r = int64_t(nh_l + 2 * nkv_l) * 128;
#pragma unroll 1
  for (int hh = 0; hh < BN / 128; ++hh) {
    const int64_t n0 = int64_t(tile_q) * BN + 128 * hh;
    if (n0 >= a.N) break;   // uniform over the CTA
    float x[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(trow + uint32_t(128 * hh + 32 * c), r);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 32; ++e) x[32 * c + e] = round_t<bf16>(__uint_as_float(r[e]));
    }
    if (!row_ok) continue;
    const int shard = int(n0 / width_r);
    const int loc = int((n0 % width_r) / 128);
    if (loc < nh_l + nkv_l) {
      const bool is_q = loc < nh_l;
      const int hidx = is_q ? shard * nh_l + loc : shard * nkv_l + (loc - nh_l);
      bf16* dst;
      if (is_q) {
        if (hidx == 0 && !pos_ok && a.err != nullptr) atomicAdd(a.err, 1);   // once per token
        dst = a.q_out + (m * a.nh + hidx) * 128;
      } else {
        if (slot == -1) continue;                                           // padding: not stored
        if (slot < 0 || slot >= a.num_slots) {
          if (hidx == 0 && a.err != nullptr) atomicAdd(a.err, 1);
          continue;
        }
        if (!pos_ok) continue;
        dst = a.k_cache + (slot * a.nkv + hidx) * 128;
      }
      float part[8];
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        float x1[8], x2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          x1[e] = x[8 * pp + e];
          x2[e] = x[64 + 8 * pp + e];
        }
        part[pp] = qk_ss8(x1, x2);
      }
      const float inv = qk_inv_rms(qk_ss_tree(part), a.eps);
      const bf16* gamma = is_q ? a.q_gamma : a.k_gamma;
      const float* cs = a.cos_sin + (pos_ok ? pos : 0) * 128;
#pragma unroll
      for (int pp = 0; pp < 8; ++pp) {
        float g1[8], g2[8], cc[8], sn[8], y1[8], y2[8];
        load16(gamma + 8 * pp, g1);
        load16(gamma + 64 + 8 * pp, g2);
        *reinterpret_cast<float4*>(cc) = *reinterpret_cast<const float4*>(cs + 8 * pp);
        *reinterpret_cast<float4*>(cc + 4) = *reinterpret_cast<const float4*>(cs + 8 * pp + 4);
        *reinterpret_cast<float4*>(sn) = *reinterpret_cast<const float4*>(cs + 64 + 8 * pp);
        *reinterpret_cast<float4*>(sn + 4) = *reinterpret_cast<const float4*>(cs + 64 + 8 * pp + 4);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          qk_rope_pair(x[8 * pp + e], x[64 + 8 * pp + e], inv, g1[e], g2[e], cc[e], sn[e], pos_ok, y1[e], y2[e]);
        store16(dst + 8 * pp, y1);
        store16(dst + 64 + 8 * pp, y2);
      }
    } else {   // v head: the rounded QKV values, a bit copy into the cache
      const int g = shard * nkv_l + (loc - nh_l - nkv_l);
      if (slot < 0 || slot >= a.num_slots || !pos_ok) continue;
      bf16* dst = a.v_cache + (slot * a.nkv + g) * 128;
#pragma unroll
      for (int v = 0; v < 16; ++v) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = x[8 * v + e];
        store16(dst + 8 * v, f);
      }
    }
  }
}

template <int BN>
struct TileCfg {
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = BN * BK * 2;
  static constexpr uint32_t TMEM_COLS = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
};

template <int BN, int STAGES>
constexpr size_t smem_bytes() {
  return 1024 + size_t(STAGES) * (TileCfg<BN>::A_BYTES + TileCfg<BN>::B_BYTES) + 256;
}

// SWAP=false: MMA-A = activations rows (M), MMA-B = weight rows (N).
// SWAP=true : MMA-A = weight rows (N),      MMA-B = token rows (M, padded to BN).
template <int BN, int STAGES, bool SWAP, int EPI, bool WROW>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmAct, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmC, TcArgs a) {
  using Cfg = TileCfg<BN>;
  constexpr uint32_t A_BYTES = Cfg::A_BYTES, B_BYTES = Cfg::B_BYTES;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t bar_done = smem_u32(bars + 2 * STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lin = blockIdx.x;
  const int tile_p = a.p_fastest ? lin % a.p_tiles : lin / a.q_tiles;
  const int tile_q = a.p_fastest ? lin / a.p_tiles : lin % a.q_tiles;
  const int split = blockIdx.y;
  const int kb0 = split * a.kblocks;
  const int kb1 = min(a.kblocks_total, kb0 + a.kblocks);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
    prefetch_map(&tmAct);
    prefetch_map(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_trigger();   // the next kernel may start its prologue
  int issued = kb0;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int r_s = 0;
    int64_t jl0 = 0;
    if (EPI == EPI_SILU) {
      const int t = SWAP ? tile_p : tile_q;
      r_s = t / a.silu_tps;
      jl0 = int64_t(t % a.silu_tps) * (SWAP ? BM / 2 : BN / 2);
    }
    // weight slab of k-block kb into ring stage s (weights are constants)
    auto load_w = [&](int kb, int s) {
      int xw, rw = 0;
      if (WROW) {
        rw = kb / a.kpb;
        xw = (kb % a.kpb) * BK;
      } else {
        xw = kb * BK;
      }
      const uint32_t dW = SWAP ? smem_u32(sA + s * A_BYTES) : smem_u32(sB + s * B_BYTES);
      const uint32_t half = SWAP ? A_BYTES / 2 : B_BYTES / 2;
      if (EPI == EPI_SILU) {
        const int64_t g0 = int64_t(r_s) * 2 * a.i_l + jl0;
        tma_load_2d(dW, &tmW, bar_full(s), xw, int(g0));
        tma_load_2d(dW + half, &tmW, bar_full(s), xw, int(g0 + a.i_l));
      } else if (WROW) {
        tma_load_3d(dW, &tmW, bar_full(s), xw, SWAP ? tile_p * BM : tile_q * BN, rw);
      } else {
        tma_load_2d(dW, &tmW, bar_full(s), xw, SWAP ? tile_p * BM : tile_q * BN);
      }
    };
    // activation slab of k-block kb (written by the previous kernel)
    auto load_act = [&](int kb, int s) {
      int xa;
      if (WROW) xa = int((kb / a.kpb) * a.k_shard) + (kb % a.kpb) * BK;
      else xa = kb * BK;
      if (!SWAP) tma_load_2d(smem_u32(sA + s * A_BYTES), &tmAct, bar_full(s), xa, tile_p * BM);
      else tma_load_2d(smem_u32(sB + s * B_BYTES), &tmAct, bar_full(s), xa, tile_q * BN);
    };
    // prologue: the first ring's weights stream in while the previous kernel finishes
    const int npre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
    for (int i = 0; i < npre; ++i) {
      mbar_expect_tx(bar_full(i), A_BYTES + B_BYTES);
      load_w(kb0 + i, i);
    }
    pdl_wait();
    for (int i = 0; i < npre; ++i) load_act(kb0 + i, i);
    issued = kb0 + npre;
    for (int kb = kb0 + npre; kb < kb1; ++kb) {
      const int i = kb - kb0;
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (!mbar_wait(bar_empty(s), ph ^ 1, 1u)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      mbar_expect_tx(bar_full(s), A_BYTES + B_BYTES);
      load_w(kb, s);
      load_act(kb, s);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    int kb = kb0;
    for (; kb < kb1; ++kb) {
      const int i = kb - kb0;
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      if (!mbar_wait(bar_full(s), ph, 2u)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint64_t da = sw128_desc(smem_u32(sA + s * A_BYTES));
      const uint64_t db = sw128_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k)
        umma_bf16(tmem, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc, (i > 0 || k > 0) ? 1u : 0u);
      umma_commit(bar_empty(s));
    }
    *consumed = kb;
    umma_commit(bar_done);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const bool ok = mbar_wait(bar_done, 0, 4u);
    tc_fence_after();
    const int quarter = warp & 3;
    const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16);
    const bool has_acc = kb1 > kb0;
    if (!SWAP) {
      const int64_t m = int64_t(tile_p) * BM + quarter * 32 + lane;
      const int64_t m0 = int64_t(tile_p) * BM + quarter * 32;   // this warp's first row
      // a.tma_store: staged in the ring's shared memory, free now that every MMA has completed
      BoxStore bs{smem_u32(sA) + uint32_t(quarter) * 2u * P_STAGE_BOX, lane};
      if (EPI == EPI_NONE && a.tma_store) {
        epi_store_tma(bs, &tmC, trow, BN, m0, a.M, int64_t(tile_q) * BN, a.N, !ok || !has_acc);
        bs.finish();
      } else if (EPI == EPI_NONE) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(trow + c, r);
          tmem_ld_wait();
          if (!ok || !has_acc) {
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = 0u;
          }
          const int64_t n0 = int64_t(tile_q) * BN + c;
          if (m < a.M) {
            bf16* dst = a.C + m * a.ldc + n0;
            if (n0 + 32 <= a.N) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 u;
                u.x = pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                u.y = pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                u.z = pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                u.w = pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                d4[v] = u;
              }
            } else {
              for (int e = 0; e < 32; ++e)
                if (n0 + e < a.N) dst[e] = __float2bfloat16_rn(__uint_as_float(r[e]));
            }
          }
        }
      } else if (EPI == EPI_ADDNORM) {
        // pass 1: the new residual s = round(round(acc) + resid) of this CTA's
        // 256 columns, written back in place, and its sum of squares (in column
        // order) left in shared memory for the cluster
        float ss = 0.0f;
        const bool row_ok = m < a.M;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(trow + c, r);
          tmem_ld_wait();
          if (!row_ok) continue;
          const int64_t n0 = int64_t(tile_q) * BN + c;
          bf16* rp = a.resid + m * a.ldc + n0;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float x[8], f[8];
            load16(rp + 8 * v, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float o = (ok && has_acc) ? round_t<bf16>(__uint_as_float(r[8 * v + e])) : 0.0f;
              f[e] = round_t<bf16>(__fadd_rn(o, x[e]));
              ss = __fadd_rn(ss, __fmul_rn(f[e], f[e]));
            }
            store16(rp + 8 * v, f);
          }
        }
        reinterpret_cast<float*>(sA)[quarter * 32 + lane] = ss;   // the ring is free: every MMA has completed
      } else if (EPI == EPI_QKV) {
        epi_qkv_tile(a, trow, m, tile_q, m < a.M && ok && has_acc);
      } else {  // EPI_SILU
        const int r_s = tile_q / a.silu_tps;
        const int64_t jl0 = int64_t(tile_q % a.silu_tps) * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(trow + c, g);
          tmem_ld32(trow + BN / 2 + c, u);
          tmem_ld_wait();
          if (m < a.M && ok && has_acc) {
            const int64_t j0 = jl0 + c;
            bf16* dst = a.C + m * a.ldc + int64_t(r_s) * a.i_l + j0;
            if (j0 + 32 <= a.i_l) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  o[e] = silu_mul_bf16(__uint_as_float(g[8 * v + e]), __uint_as_float(u[8 * v + e]));
                uint4 w;
                w.x = pack_bf16(o[0], o[1]);
                w.y = pack_bf16(o[2], o[3]);
                w.z = pack_bf16(o[4], o[5]);
                w.w = pack_bf16(o[6], o[7]);
                d4[v] = w;
              }
            } else {
              for (int e = 0; e < 32; ++e)
                if (j0 + e < a.i_l)
                  dst[e] = __float2bfloat16_rn(silu_mul_bf16(__uint_as_float(g[e]), __uint_as_float(u[e])));
            }
          }
        }
      }
    } else {
      // swapped: TMEM lane = weight row of the tile, column = token
      const int pl = quarter * 32 + lane;
      const int mv = int(a.M);   // tokens (<= BN)
      const int64_t p = int64_t(tile_p) * BM + pl;
      float* part_s = reinterpret_cast<float*>(sA);   // ring slots are free once the MMAs are done
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        uint32_t r[32];
        tmem_ld32(trow + c, r);   // TMEM_COLS >= 32 >= BN - c: the load stays inside the allocation
        tmem_ld_wait();
        if (!ok || !has_acc) {
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = 0u;
        }
        const int lim = BN - c < 32 ? BN - c : 32;
        if (a.splits == 1 && EPI == EPI_NONE) {
          if (p < a.N)
            for (int e = 0; e < lim; ++e)
              if (c + e < mv) a.C[int64_t(c + e) * a.ldc + p] = __float2bfloat16_rn(__uint_as_float(r[e]));
        } else {
          for (int e = 0; e < lim; ++e) part_s[(c + e) * BM + pl] = __uint_as_float(r[e]);
        }
      }
    }
  }

  if (!SWAP && EPI == EPI_ADDNORM) {
    // the row's sum of squares over the cluster's CTAs (rank order), then pass 2:
    // y = round(s * rsqrt(mean(s^2) + eps) * gamma) over this CTA's columns
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2) {
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const int64_t m = int64_t(tile_p) * BM + row;
      const uint32_t base = smem_u32(sA) + uint32_t(row) * 4u;
      float tot = 0.0f;
      for (int r = 0; r < a.q_tiles; ++r) tot = __fadd_rn(tot, ld_cluster_f32(map_to_rank(base, uint32_t(r))));
      const float inv = rsqrtf(__fadd_rn(__fdiv_rn(tot, float(a.N)), a.eps));
      if (m < a.M) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 8) {
          const int64_t n0 = int64_t(tile_q) * BN + c;
          float x[8], g[8], y[8];
          load16(a.resid + m * a.ldc + n0, x);
          load16(a.norm_gamma + n0, g);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), g[e]);
          store16(a.y_out + m * a.ldc + n0, y);
        }
      }
    }
    // keep every CTA's shared memory alive until all ranks have read it
    cluster_sync_all();
  }

  if (SWAP && (a.splits > 1 || EPI == EPI_SILU)) {
    // every CTA of the cluster has its partial tile in shared memory (a lone
    // CTA is a cluster of one)
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2) {
      // reduce-scatter: rank r sums the splits for the tile rows f = r, r + S, ...
      // (SiluAndMul: gate row f and up row f + 64) and writes those outputs
      const int S = a.splits;
      const uint32_t rank = cluster_rank();
      const int mv = int(a.M);
      const int te = threadIdx.x - 64;                 // 0..127 over the epilogue warps
      constexpr int NF = EPI == EPI_SILU ? BM / 2 : BM;
      const int nf_mine = (NF - int(rank) + S - 1) / S;
      const uint32_t base = smem_u32(sA);
      uint32_t peer[kMaxCluster];
#pragma unroll
      for (int sp = 0; sp < kMaxCluster; ++sp) peer[sp] = sp < S ? map_to_rank(base, uint32_t(sp)) : 0u;
      const int total = nf_mine * mv;
#pragma unroll 2
      for (int idx = te; idx < total; idx += 128) {
        const int fi = idx % nf_mine, j = idx / nf_mine;
        const int f = int(rank) + S * fi;
        const uint32_t off_g = uint32_t(j * BM + f) * 4u;
        float vg[kMaxCluster], vu[kMaxCluster];
#pragma unroll
        for (int sp = 0; sp < kMaxCluster; ++sp) {
          vg[sp] = sp < S ? ld_cluster_f32(peer[sp] + off_g) : 0.0f;
          if (EPI == EPI_SILU) vu[sp] = sp < S ? ld_cluster_f32(peer[sp] + off_g + uint32_t(BM / 2) * 4u) : 0.0f;
        }
        float g = 0.0f, u = 0.0f;
#pragma unroll
        for (int sp = 0; sp < kMaxCluster; ++sp)
          if (sp < S) {   // split order: deterministic
            g += vg[sp];
            if (EPI == EPI_SILU) u += vu[sp];
          }
        if (EPI == EPI_NONE) {
          const int64_t pcol = int64_t(tile_p) * BM + f;
          if (pcol < a.N) a.C[int64_t(j) * a.ldc + pcol] = __float2bfloat16_rn(g);
        } else {
          const int r_s = tile_p / a.silu_tps;
          const int64_t jl = int64_t(tile_p % a.silu_tps) * (BM / 2) + f;
          if (jl < a.i_l) a.C[int64_t(j) * a.ldc + int64_t(r_s) * a.i_l + jl] = __float2bfloat16_rn(silu_mul_bf16(g, u));
        }
      }
    }
    // keep every CTA's shared memory alive until all ranks have read it
    cluster_sync_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // drain copies that were issued but never consumed, so that no TMA write
    // lands in shared memory after the CTA exits
    for (int kb = *consumed; kb < issued; ++kb) {
      const int i = kb - kb0;
      mbar_wait(bar_full(i % STAGES), (i / STAGES) & 1, 8u);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// 256 x 256 prefill tiles.  A CTA covers 256 token rows as two 128-row MMA
// halves that share every weight slab: per 64-wide k-block, 32 KB of
// activations and 32 KB of weights feed 2 x 128 x 256 x 64 MACs.  That is 1.5
// times the work per byte of a 128 x 256 tile, for GEMMs bound by L2 -> SM
// operand traffic.  TMEM holds both accumulators (all 512 columns); the TMA
// ring has 3 stages of 64 KB; one tile per CTA.  Same producer / MMA roles as
// gemm_tc_kernel, with two epilogue warpgroups draining the halves side by side.
constexpr int M2_THREADS = 320;
// ---------------------------------------------------------------------------
constexpr int M2_ROWS = 256, M2_STAGES = 3;
constexpr uint32_t M2_A_BYTES = M2_ROWS * BK * 2, M2_B_BYTES = 256 * BK * 2;
constexpr size_t m2_smem_bytes() { return 1024 + size_t(M2_STAGES) * (M2_A_BYTES + M2_B_BYTES) + 256; }

template <int EPI, bool WROW>
__global__ void __launch_bounds__(M2_THREADS, 1)
    gemm_tc_m256_kernel(const __grid_constant__ CUtensorMap tmAct, const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmC, TcArgs a) {
  static_assert(EPI == EPI_NONE || EPI == EPI_SILU || EPI == EPI_ADDNORM, "plain, SiluAndMul or add + RMSNorm");
  constexpr int BN = 256, STAGES = M2_STAGES;
  constexpr uint32_t A_BYTES = M2_A_BYTES, B_BYTES = M2_B_BYTES, TMEM_COLS = 512;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + STAGES * A_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  const uint32_t bar_done = smem_u32(bars + 2 * STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lin = blockIdx.x;
  const int tile_p = a.p_fastest ? lin % a.p_tiles : lin / a.q_tiles;   // 256-row block
  const int tile_q = a.p_fastest ? lin / a.p_tiles : lin % a.q_tiles;
  const int nk = a.kblocks_total;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
    prefetch_map(&tmAct);
    prefetch_map(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_trigger();   // the next kernel may start its prologue
  int issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    int r_s = 0;
    int64_t jl0 = 0;
    if (EPI == EPI_SILU) {
      r_s = tile_q / a.silu_tps;
      jl0 = int64_t(tile_q % a.silu_tps) * (BN / 2);
    }
    auto load_w = [&](int kb, int s) {   // weight slab (constants)
      int xw, rw = 0;
      if (WROW) {
        rw = kb / a.kpb;
        xw = (kb % a.kpb) * BK;
      } else {
        xw = kb * BK;
      }
      const uint32_t dW = smem_u32(sB + s * B_BYTES);
      if (EPI == EPI_SILU) {
        const int64_t g0 = int64_t(r_s) * 2 * a.i_l + jl0;
        tma_load_2d(dW, &tmW, bar_full(s), xw, int(g0));
        tma_load_2d(dW + B_BYTES / 2, &tmW, bar_full(s), xw, int(g0 + a.i_l));
      } else if (WROW) {
        tma_load_3d(dW, &tmW, bar_full(s), xw, tile_q * BN, rw);
      } else {
        tma_load_2d(dW, &tmW, bar_full(s), xw, tile_q * BN);
      }
    };
    auto load_act = [&](int kb, int s) {   // 256 activation rows (written by the previous kernel)
      const int xa = WROW ? int((kb / a.kpb) * a.k_shard) + (kb % a.kpb) * BK : kb * BK;
      tma_load_2d(smem_u32(sA + s * A_BYTES), &tmAct, bar_full(s), xa, tile_p * M2_ROWS);
    };
    const int npre = nk < STAGES ? nk : STAGES;
    for (int i = 0; i < npre; ++i) {
      mbar_expect_tx(bar_full(i), A_BYTES + B_BYTES);
      load_w(i, i);
    }
    pdl_wait();
    for (int i = 0; i < npre; ++i) load_act(i, i);
    issued = npre;
    for (int kb = npre; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait(bar_empty(s), ph ^ 1, 1u)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      mbar_expect_tx(bar_full(s), A_BYTES + B_BYTES);
      load_w(kb, s);
      load_act(kb, s);
      issued = kb + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer: two 128-row halves per weight slab ----------------
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    int kb = 0;
    for (; kb < nk; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      if (!mbar_wait(bar_full(s), ph, 2u)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint64_t da0 = sw128_desc(smem_u32(sA + s * A_BYTES));
      const uint64_t da1 = sw128_desc(smem_u32(sA + s * A_BYTES) + uint32_t(BM) * 128u);   // rows 128 .. 255
      const uint64_t db = sw128_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
      for (int k = 0; k < BK / UMMA_K; ++k) {
        umma_bf16(tmem, da0 + uint64_t(2 * k), db + uint64_t(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        umma_bf16(tmem + uint32_t(BN), da1 + uint64_t(2 * k), db + uint64_t(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(bar_empty(s));
    }
    *consumed = kb;
    umma_commit(bar_done);
  } else if (warp >= 2) {
    // ---------------- epilogue: warps 2-5 drain half 0, warps 6-9 half 1 ----------------
    const bool ok = mbar_wait(bar_done, 0, 4u);
    tc_fence_after();
    const int quarter = warp & 3;   // TMEM lanes this warp may access
    const int h = (warp - 2) >> 2;
    const bool zero = !ok || nk <= 0;
    // staging boxes in the drained ring, two per warp
    BoxStore bs{smem_u32(sA) + uint32_t(warp - 2) * 2u * P_STAGE_BOX, lane};
    {
      const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(h * BN);
      const int64_t m0 = int64_t(tile_p) * M2_ROWS + h * BM + quarter * 32;   // this warp's first row
      if (EPI == EPI_NONE) {
        if (a.tma_store) epi_store_tma(bs, &tmC, trow, BN, m0, a.M, int64_t(tile_q) * BN, a.N, zero);
        else epi_store_direct(trow, BN, m0 + lane, a, int64_t(tile_q) * BN, zero);
      } else if (EPI == EPI_ADDNORM) {
        // pass 1: the new residual s = round(round(acc) + resid) of this CTA's 256
        // columns, written back in place, and its sum of squares (in column order)
        // left in shared memory for the cluster (the ring is free: every MMA has completed)
        const int64_t m = m0 + lane;
        float ss = 0.0f;
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(trow + c, r);
          tmem_ld_wait();
          if (m >= a.M) continue;
          bf16* rp = a.resid + m * a.ldc + int64_t(tile_q) * BN + c;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            float x[8], f[8];
            load16(rp + 8 * v, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float o = zero ? 0.0f : round_t<bf16>(__uint_as_float(r[8 * v + e]));
              f[e] = round_t<bf16>(__fadd_rn(o, x[e]));
              ss = __fadd_rn(ss, __fmul_rn(f[e], f[e]));
            }
            store16(rp + 8 * v, f);
          }
        }
        reinterpret_cast<float*>(sA)[h * BM + quarter * 32 + lane] = ss;
      } else {
        epi_silu_direct(trow, BN / 2, m0 + lane, a, tile_q / a.silu_tps, int64_t(tile_q % a.silu_tps) * (BN / 2), !zero);
      }
    }
    if (EPI == EPI_NONE) bs.finish();
  }

  if (EPI == EPI_ADDNORM) {
    // the row's sum of squares over the cluster's CTAs (rank order), then pass 2:
    // y = round(s * rsqrt(mean(s^2) + eps) * gamma) over this CTA's columns
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2) {
      const int row = ((warp - 2) >> 2) * BM + (warp & 3) * 32 + lane;
      const int64_t m = int64_t(tile_p) * M2_ROWS + row;
      const uint32_t base = smem_u32(sA) + uint32_t(row) * 4u;
      float tot = 0.0f;
      for (int r = 0; r < a.q_tiles; ++r) tot = __fadd_rn(tot, ld_cluster_f32(map_to_rank(base, uint32_t(r))));
      const float inv = rsqrtf(__fadd_rn(__fdiv_rn(tot, float(a.N)), a.eps));
      if (m < a.M) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 8) {
          const int64_t n0 = int64_t(tile_q) * BN + c;
          float x[8], g[8], y[8];
          load16(a.resid + m * a.ldc + n0, x);
          load16(a.norm_gamma + n0, g);
#pragma unroll
          for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(x[e], inv), g[e]);
          store16(a.y_out + m * a.ldc + n0, y);
        }
      }
    }
    // keep every CTA's shared memory alive until all ranks have read it
    cluster_sync_all();
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // drain copies that were issued but never consumed
    for (int kb = *consumed; kb < issued; ++kb) mbar_wait(bar_full(kb % STAGES), (kb / STAGES) & 1, 8u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent prefill GEMM (many tokens: MMA-A = activations, MMA-B = weights,
// 128 x 256 tiles, no K split).  One CTA per SM walks the tiles blockIdx.x,
// blockIdx.x + gridDim.x, ...  The TMA ring runs on across tile boundaries,
// and TMEM holds two 128 x 256 fp32 accumulators (all 512 columns): the
// epilogue warps drain tile j from one buffer while the MMA thread
// accumulates tile j + 1 into the other, so neither the pipeline fill nor
// the epilogue of a tile leaves the tensor cores idle.
//
// Barriers: full[s] / empty[s] per ring stage (TMA bytes landed / MMAs done
// reading); acc_full[b] (MMA commit: the tile in buffer b is complete) and
// acc_empty[b] (one arrival per epilogue warp: buffer b has been read out);
// drain (the MMA thread's last commit, so that no MMA is in flight at exit).
// Ring iteration `it` counts (tile, k-block) pairs of this CTA: stage it % S,
// phase parity (it / S) & 1.  The u-th use of accumulator b (tile j = 2u + b)
// waits for acc_empty completion u - 1 (parity (u & 1) ^ 1, which a fresh
// barrier satisfies for u = 0) and the epilogue waits for acc_full
// completion u (parity u & 1).
// ---------------------------------------------------------------------------
constexpr int PBN = 256, PSTAGES = 4;
constexpr uint32_t P_TMEM_COLS = 512;
// epilogue staging (BoxStore): two boxes per epilogue warp, 1 KB past the ring's barrier area
constexpr size_t psmem_bytes() {
  return 1024 + size_t(PSTAGES) * (TileCfg<PBN>::A_BYTES + TileCfg<PBN>::B_BYTES) + 1024 + 4 * 2 * P_STAGE_BOX;
}

template <int EPI, bool WROW>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_persist_kernel(const __grid_constant__ CUtensorMap tmAct, const __grid_constant__ CUtensorMap tmW,
                           const __grid_constant__ CUtensorMap tmC, TcArgs a) {
  constexpr int BN = PBN, STAGES = PSTAGES;
  constexpr uint32_t A_BYTES = TileCfg<BN>::A_BYTES, B_BYTES = TileCfg<BN>::B_BYTES;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = sm;
  uint8_t* sB = sm + STAGES * A_BYTES;
  // full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * B_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* consumed = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar_full = [&](int s) { return smem_u32(bars + s); };
  auto bar_empty = [&](int s) { return smem_u32(bars + STAGES + s); };
  auto bar_acc_full = [&](int b) { return smem_u32(bars + 2 * STAGES + b); };
  auto bar_acc_empty = [&](int b) { return smem_u32(bars + 2 * STAGES + 2 + b); };
  const uint32_t bar_drain = smem_u32(bars + 2 * STAGES + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tiles = a.p_tiles * a.q_tiles;   // the host keeps this and `total` inside int
  const int bx = int(blockIdx.x), gx = int(gridDim.x);
  const int my_tiles = bx < n_tiles ? (n_tiles - bx + gx - 1) / gx : 0;
  const int nk = a.kblocks_total;
  const int total = my_tiles * nk;   // ring iterations of this CTA
  auto tile_of = [&](int j, int& tile_p, int& tile_q) {
    const int t = bx + j * gx;
    tile_p = a.p_fastest ? t % a.p_tiles : t / a.q_tiles;
    tile_q = a.p_fastest ? t / a.p_tiles : t % a.q_tiles;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_acc_full(b), 1);
      mbar_init(bar_acc_empty(b), 4);   // one arrival per epilogue warp
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    *consumed = 0;
    fence_mbar_init();
    prefetch_map(&tmAct);
    prefetch_map(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), P_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_trigger();   // the next kernel may start its prologue
  int issued = 0;
  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    // ring iteration it: the weight slab (w) and/or activation slab (act) of
    // its k-block into stage s
    auto load = [&](int it, int s, bool w, bool act) {
      const int j = it / nk, kb = it - j * nk;
      int tile_p, tile_q;
      tile_of(j, tile_p, tile_q);
      if (w) {
        int xw, rw = 0;
        if (WROW) {
          rw = kb / a.kpb;
          xw = (kb % a.kpb) * BK;
        } else {
          xw = kb * BK;
        }
        const uint32_t dW = smem_u32(sB + s * B_BYTES);
        if (EPI == EPI_SILU) {
          // 128 gate rows then the matching 128 up rows of shard r_s
          const int r_s = tile_q / a.silu_tps;
          const int64_t g0 = int64_t(r_s) * 2 * a.i_l + int64_t(tile_q % a.silu_tps) * (BN / 2);
          tma_load_2d(dW, &tmW, bar_full(s), xw, int(g0));
          tma_load_2d(dW + B_BYTES / 2, &tmW, bar_full(s), xw, int(g0 + a.i_l));
        } else if (WROW) {
          tma_load_3d(dW, &tmW, bar_full(s), xw, tile_q * BN, rw);
        } else {
          tma_load_2d(dW, &tmW, bar_full(s), xw, tile_q * BN);
        }
      }
      if (act) {
        const int xa = WROW ? int((kb / a.kpb) * a.k_shard) + (kb % a.kpb) * BK : kb * BK;
        tma_load_2d(smem_u32(sA + s * A_BYTES), &tmAct, bar_full(s), xa, tile_p * BM);
      }
    };
    // the first ring's weights (constants) stream in while the previous kernel finishes
    const int npre = total < STAGES ? total : STAGES;
    for (int i = 0; i < npre; ++i) {
      mbar_expect_tx(bar_full(i), A_BYTES + B_BYTES);
      load(i, i, true, false);
    }
    pdl_wait();
    for (int i = 0; i < npre; ++i) load(i, i, false, true);
    issued = npre;
    for (int it = npre; it < total; ++it) {
      const int s = it % STAGES;
      const uint32_t ph = uint32_t(it / STAGES) & 1u;
      if (!mbar_wait(bar_empty(s), ph ^ 1u, 1u)) {
        *abort_flag = 1;
        break;
      }
      if (*abort_flag) break;
      mbar_expect_tx(bar_full(s), A_BYTES + B_BYTES);
      load(it, s, true, true);
      issued = it + 1;
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16(BM, BN);
    int it = 0;
    for (int j = 0; j < my_tiles; ++j) {
      const int b = j & 1;
      const uint32_t use = uint32_t(j >> 1) & 1u;
      if (*abort_flag) break;
      if (!mbar_wait(bar_acc_empty(b), use ^ 1u, 2u)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t d = tmem + uint32_t(b * BN);
      bool stop = false;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = uint32_t(it / STAGES) & 1u;
        if (!mbar_wait(bar_full(s), ph, 2u)) {
          *abort_flag = 1;
          stop = true;
          break;
        }
        tc_fence_after();
        const uint64_t da = sw128_desc(smem_u32(sA + s * A_BYTES));
        const uint64_t db = sw128_desc(smem_u32(sB + s * B_BYTES));
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k)
          umma_bf16(d, da + uint64_t(2 * k), db + uint64_t(2 * k), idesc, (kb > 0 || k > 0) ? 1u : 0u);
        umma_commit(bar_empty(s));
        *consumed = it + 1;
      }
      if (stop) break;
      umma_commit(bar_acc_full(b));
    }
    // past this wait no MMA of this CTA is in flight (nor reads shared memory)
    umma_commit(bar_drain);
    mbar_wait(bar_drain, 0, 8u);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    // waits and the abort check are warp-uniform: tcgen05.ld is .sync.aligned
    const int quarter = warp & 3;
    // a.tma_store: stores through tmC (BoxStore)
    BoxStore bs{smem_u32(sm) + uint32_t(STAGES) * (A_BYTES + B_BYTES) + 1024u + uint32_t(quarter) * 2u * P_STAGE_BOX,
                lane};
    for (int j = 0; j < my_tiles; ++j) {
      const int b = j & 1;
      const uint32_t use = uint32_t(j >> 1) & 1u;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(bar_acc_full(b), use, 4u));
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      tc_fence_after();
      int tile_p, tile_q;
      tile_of(j, tile_p, tile_q);
      const uint32_t trow = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(b * BN);
      const int64_t m = int64_t(tile_p) * BM + quarter * 32 + lane;
      const int64_t m0 = int64_t(tile_p) * BM + quarter * 32;   // this warp's first row
      if (EPI == EPI_NONE && a.tma_store) {
        epi_store_tma(bs, &tmC, trow, BN, m0, a.M, int64_t(tile_q) * BN, a.N, false);
      } else if (EPI == EPI_SILU && a.tma_store) {
        const int r_s = tile_q / a.silu_tps;
        const int64_t jl0 = int64_t(tile_q % a.silu_tps) * (BN / 2);
        epi_silu_tma(bs, &tmC, trow, BN / 2, m0, a.M, int64_t(r_s) * a.i_l + jl0, jl0, a.i_l, false);
      } else if (EPI == EPI_NONE) {
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(trow + c, r);
          tmem_ld_wait();
          const int64_t n0 = int64_t(tile_q) * BN + c;
          if (m < a.M) {
            bf16* dst = a.C + m * a.ldc + n0;
            if (n0 + 32 <= a.N) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 u;
                u.x = pack_bf16(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1]));
                u.y = pack_bf16(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3]));
                u.z = pack_bf16(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5]));
                u.w = pack_bf16(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7]));
                d4[v] = u;
              }
            } else {
              for (int e = 0; e < 32; ++e)
                if (n0 + e < a.N) dst[e] = __float2bfloat16_rn(__uint_as_float(r[e]));
            }
          }
        }
      } else if (EPI == EPI_QKV) {
        epi_qkv_tile(a, trow, m, tile_q, m < a.M);
      } else {  // EPI_SILU: columns [0, 128) gate, [128, 256) up
        const int r_s = tile_q / a.silu_tps;
        const int64_t jl0 = int64_t(tile_q % a.silu_tps) * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t g[32], u[32];
          tmem_ld32(trow + c, g);
          tmem_ld32(trow + BN / 2 + c, u);
          tmem_ld_wait();
          if (m < a.M) {
            const int64_t j0 = jl0 + c;
            bf16* dst = a.C + m * a.ldc + int64_t(r_s) * a.i_l + j0;
            if (j0 + 32 <= a.i_l) {
              uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                float o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  o[e] = silu_mul_bf16(__uint_as_float(g[8 * v + e]), __uint_as_float(u[8 * v + e]));
                uint4 w;
                w.x = pack_bf16(o[0], o[1]);
                w.y = pack_bf16(o[2], o[3]);
                w.z = pack_bf16(o[4], o[5]);
                w.w = pack_bf16(o[6], o[7]);
                d4[v] = w;
              }
            } else {
              for (int e = 0; e < 32; ++e)
                if (j0 + e < a.i_l)
                  dst[e] = __float2bfloat16_rn(silu_mul_bf16(__uint_as_float(g[e]), __uint_as_float(u[e])));
            }
          }
        }
      }
      // this warp's 32 accumulator lanes are read out: hand the buffer back
      tc_fence_before();
      __syncwarp();
      if (lane == 0) tcx::mbar_arrive(bar_acc_empty(b));
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
    }
    bs.finish();   // the tensor stores are complete before the CTA exits
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // drain copies that were issued but never consumed, so that no TMA write
    // lands in shared memory after the CTA exits
    for (int i = *consumed; i < issued; ++i) mbar_wait(bar_full(i % STAGES), uint32_t(i / STAGES) & 1u, 8u);
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, P_TMEM_COLS);
  }
}

// The bounded-wait path of the tensor-core kernels, run on purpose: one
// thread waits on a fresh mbarrier for a phase that nothing completes.  After
// the time limit the wait records kSelftestCode in the error word and the
// kernel returns, leaving the context usable; qw_device_error reports it.
constexpr uint32_t kSelftestCode = 0x100u;

__global__ void __launch_bounds__(32) selftest_wait_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);   // one arrival completes phase 0, and none is made
  fence_mbar_init();
  mbar_wait(b, 0, kSelftestCode);
}

}  // namespace tc

// ===========================================================================
// Few-token GEMM (decode): weight streaming with warp-level MMA.
//
// C[M, N] = A[M, K] W^T for M <= 64.  The weights are read once and dominate
// the bytes, so the kernel is built for memory-level parallelism: a CTA owns
// 16 weight rows (SiluAndMul: 8 gate rows and the matching 8 up rows; 8 rows
// for narrow outputs above 8 tokens) across the whole K, split over its 8
// warps.  The weights are constants, so their transfer starts before the
// programmatic dependency wait: up to 8 tokens (WTMA) as bulk copies of
// whole rows into shared memory, otherwise as 16-byte non-caching loads into
// registers issued up front by each warp.  The MMAs are mma.sync m16n8k16.  Weights and tokens use the same permutation of the 32
// k values of a chunk (thread t holds k 8t..8t+7: logical k 2t,2t+1 | 2t+8,2t+9
// of two k-steps), so no shuffles are needed.  The 8 warps' partial tiles are
// added in shared memory in warp order (deterministic) and the epilogue
// writes bf16 (or silu(gate) * up).
// ===========================================================================
constexpr int GV_WARPS = 8;

__device__ __forceinline__ uint4 ldg_stream(const bf16* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// RPC: weight rows per CTA (16, or 8 for small N to spread over more SMs);
// MAXC: 32-wide k chunks per warp held in registers at once.
// NORM: A is a sublayer output h; the GEMM input is y = RMSNorm(h + res_in)
// * gamma (h alone when res_in is null), computed by every CTA for all M
// tokens into shared memory; CTA 0 writes res_out = h + res_in (the new
// residual, a buffer distinct from h and res_in).
struct NormArgs {
  const bf16* res_in;
  bf16* res_out;
  const bf16* gamma;
  float eps;
};
constexpr int GV_YPAD = 8;   // y row padding (elements): 16-byte rows at distinct bank groups
// WTMA weight rows in shared memory: stride K + gv_wpad(K) elements, an odd
// multiple of 64 bytes, so the two rows a quarter-warp's 16-byte reads touch
// fall in opposite halves of the banks (K % 32 == 0)
__host__ __device__ constexpr int gv_wpad(int K) { return K % 64 == 0 ? 32 : 0; }
// byte offset of the WTMA weight rows: after the staged or normed activation rows
__host__ __device__ constexpr size_t gv_wsm_offset(int M, int K, bool norm, bool stage) {
  return (norm || stage) ? size_t(M) * (K + GV_YPAD) * 2 : 0;
}

// TL: m16 row tiles per CTA (2: SiluAndMul with 16 outputs per CTA, or 32
// plain output rows; half the CTAs, so a norm prologue runs in one wave and
// its activation reads are shared by twice the weight rows).
// STAGE: A [M][K] is copied into shared memory first, one bulk copy (TMA
// unit) per token row completing on an mbarrier, all in flight at once
// (otherwise each k chunk's activations are one more L2 round trip before its
// MMAs; per-thread 16-byte asynchronous copies queue behind the weight loads).
// WTMA: the CTA's weight rows are bulk-copied into shared memory before the
// dependency wait (one copy per row, or per shard piece of a row-split
// weight) instead of being loaded into registers by every thread; the MMAs
// then read them from shared memory.
template <int NT, int EPI, bool WROW, int RPC, int MAXC, bool NORM = false, int TL = 1, bool STAGE = false,
          bool WTMA = false>
__global__ void __launch_bounds__(GV_WARPS * 32, MAXC <= 4 ? 2 : 1)
    gemv_mma_kernel(const bf16* __restrict__ A, const bf16* __restrict__ W, bf16* __restrict__ C, int M, int N, int K,
                    int K_l, int64_t ldc, int64_t i_l, NormArgs na) {
  static_assert(TL == 1 || EPI == tc::EPI_SILU || (RPC == 16 && !WROW), "two row tiles: SiluAndMul or 16-row tiles");
  constexpr int GV_MAXC = MAXC;
  __shared__ float red[GV_WARPS][16 * TL][NT * 8];
  extern __shared__ __align__(16) uint8_t gv_dyn[];
  bf16* ys = reinterpret_cast<bf16*>(gv_dyn);   // NORM, STAGE: [M][K + GV_YPAD]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  // the two weight rows of this thread in each row tile (m16 tile rows g and g + 8)
  int64_t rowA[TL], rowB[TL];
  bool okA[TL], okB[TL];
#pragma unroll
  for (int tl = 0; tl < TL; ++tl) {
    if (EPI == tc::EPI_SILU) {
      const int64_t o0 = (int64_t(blockIdx.x) * TL + tl) * 8;   // first output column of the tile
      const int64_t r = o0 / i_l, j = o0 % i_l + g;
      rowA[tl] = r * 2 * i_l + j;                                // gate row
      rowB[tl] = rowA[tl] + i_l;                                 // matching up row
      okA[tl] = okB[tl] = (o0 + g) < int64_t(N / 2) && j < i_l;
    } else {
      rowA[tl] = (int64_t(blockIdx.x) * TL + tl) * RPC + g;
      rowB[tl] = rowA[tl] + 8;
      okA[tl] = rowA[tl] < N;
      okB[tl] = RPC == 16 && rowB[tl] < N;
    }
  }
  const int kw = ((K + GV_WARPS * 32 - 1) / (GV_WARPS * 32)) * 32;   // k values per warp, whole chunks
  const int k0 = warp * kw;
  const int k1 = min(K, k0 + kw);
  auto wptr = [&](int64_t row, int k) -> const bf16* {
    if (WROW) {
      const int r = k / K_l;
      return W + (int64_t(r) * N + row) * K_l + (k - r * K_l);
    }
    return W + row * int64_t(K) + k;
  };
  float acc[TL][NT][4];
#pragma unroll
  for (int tl = 0; tl < TL; ++tl)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[tl][n][0] = acc[tl][n][1] = acc[tl][n][2] = acc[tl][n][3] = 0.0f;
  // WTMA: local row 16 tl + g holds rowA[tl], 16 tl + 8 + g holds rowB[tl]
  const int ws_stride = K + gv_wpad(K);
  const bf16* wsm = reinterpret_cast<const bf16*>(gv_dyn + gv_wsm_offset(M, K, NORM, STAGE));
  uint4 wa[TL][GV_MAXC], wb[TL][GV_MAXC];
  auto load_w = [&](int kb) {
#pragma unroll
    for (int tl = 0; tl < TL; ++tl)
#pragma unroll
      for (int c = 0; c < GV_MAXC; ++c) {
        const int k = kb + 32 * c + 8 * t;
        const bool in = kb + 32 * c < k1;
        if (WTMA) {
          wa[tl][c] = (in && okA[tl]) ? *reinterpret_cast<const uint4*>(wsm + (16 * tl + g) * ws_stride + k)
                                      : make_uint4(0, 0, 0, 0);
          wb[tl][c] = (RPC == 16 && in && okB[tl])
                          ? *reinterpret_cast<const uint4*>(wsm + (16 * tl + 8 + g) * ws_stride + k)
                          : make_uint4(0, 0, 0, 0);
        } else {
          wa[tl][c] = (in && okA[tl]) ? ldg_stream(wptr(rowA[tl], k)) : make_uint4(0, 0, 0, 0);
          wb[tl][c] = (RPC == 16 && in && okB[tl]) ? ldg_stream(wptr(rowB[tl], k)) : make_uint4(0, 0, 0, 0);
        }
      }
  };
  __shared__ uint64_t stage_bar;   // STAGE: completion of the activation copies
  if (STAGE) {
    if (threadIdx.x == 0) {
      tcx::mbar_init(smem_u32(&stage_bar), 1);
      tcx::fence_mbar_init();
      tcx::mbar_expect_tx(smem_u32(&stage_bar), uint32_t(M) * uint32_t(K) * 2u);   // before any copy is issued
    }
    __syncthreads();
  }
  __shared__ uint64_t w_bar;   // WTMA: completion of the weight rows' copies
  if (WTMA) {
    // global row of local weight row lr (its tile, half and m16 row); false past the outputs
    auto w_row = [&](int lr, int64_t& row) -> bool {
      const int tl = lr >> 4, h = (lr >> 3) & 1, gg = lr & 7;
      if (EPI == tc::EPI_SILU) {
        const int64_t o0 = (int64_t(blockIdx.x) * TL + tl) * 8;
        const int64_t r = o0 / i_l, j = o0 % i_l + gg;
        row = r * 2 * i_l + j + (h ? i_l : 0);
        return (o0 + gg) < int64_t(N / 2) && j < i_l;
      }
      row = (int64_t(blockIdx.x) * TL + tl) * RPC + 8 * h + gg;
      return row < N && (h == 0 || RPC == 16);
    };
    constexpr int NROWS = (EPI == tc::EPI_SILU || RPC == 16 ? 16 : 8) * TL;
    const uint32_t wb_ = smem_u32(&w_bar);
    if (threadIdx.x == 0) {
      uint32_t bytes = 0;
      for (int lr = 0; lr < NROWS; ++lr) {
        int64_t row;
        if (w_row(lr, row)) bytes += uint32_t(K) * 2u;
      }
      tcx::mbar_init(wb_, 1);
      tcx::fence_mbar_init();
      tcx::mbar_expect_tx(wb_, bytes);   // <= 32 rows x 2K bytes, far below the 2^20 - 1 limit
    }
    __syncthreads();
    // the weights are constants: their copies start before the dependency wait
    if (lane == 0)
      for (int lr = warp; lr < NROWS; lr += GV_WARPS) {
        int64_t row;
        if (!w_row(lr, row)) continue;
        const uint32_t dst = smem_u32(wsm + lr * ws_stride);
        const int pieces = WROW ? K / K_l : 1;
        const int len = WROW ? K_l : K;
        for (int q = 0; q < pieces; ++q)
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                           dst + uint32_t(q * len) * 2u),
                       "l"(WROW ? W + (int64_t(q) * N + row) * K_l : W + row * int64_t(K)), "r"(uint32_t(len) * 2u),
                       "r"(wb_)
                       : "memory");
      }
  } else if (k0 < k1) {
    load_w(k0);   // the first weights are constants: loaded before the dependency wait
  }
  pdl_wait();      // the activations are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  const int ys_stride = K + GV_YPAD;
  if (NORM) {
    // y = RMSNorm(h + res_in) * gamma for every token, into shared memory.
    // h and res_in are read by plain loads: with the weight rows on bulk
    // copies the load path is free (bulk copies of these rows queue behind
    // the weights': 117.8-118.5 against 118.8-119.1 ms per 128 decode steps).
    for (int tk = warp; tk < M; tk += GV_WARPS) {
      const bf16* hr = A + int64_t(tk) * K;
      const bf16* rr = na.res_in != nullptr ? na.res_in + int64_t(tk) * K : nullptr;
      float ss = 0.0f;
      for (int k0v = lane * 8; k0v < K; k0v += 4 * 256) {
        uint4 hv[4], rv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {   // a pass's loads all in flight before use
          const int k = k0v + i * 256;
          if (k < K) {
            hv[i] = __ldcg(reinterpret_cast<const uint4*>(hr + k));
            if (rr != nullptr) rv[i] = __ldcg(reinterpret_cast<const uint4*>(rr + k));
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = k0v + i * 256;
          if (k >= K) continue;
          float v[8];
          const bf16* hb = reinterpret_cast<const bf16*>(&hv[i]);
          const bf16* rb = reinterpret_cast<const bf16*>(&rv[i]);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            v[e] = rr != nullptr ? round_t<bf16>(__bfloat162float(hb[e]) + __bfloat162float(rb[e]))
                                 : __bfloat162float(hb[e]);   // x + residual, in the model dtype
          if (na.res_out != nullptr && blockIdx.x == 0) store16(na.res_out + int64_t(tk) * K + k, v);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
          store16(ys + tk * ys_stride + k, v);   // the sum, normalised below
        }
      }
      ss = warp_sum(ss);
      const float inv = rsqrtf(ss / float(K) + na.eps);
      __syncwarp();
      for (int k = lane * 8; k < K; k += 256) {
        float v[8], gm[8];
        load16(ys + tk * ys_stride + k, v);
        load16(na.gamma + k, gm);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (v[e] * inv) * gm[e];
        store16(ys + tk * ys_stride + k, v);
      }
    }
    __syncthreads();
  }
  if (STAGE) {
    // rows of 2K bytes (K % 32 == 0) to 16-byte aligned rows of ys, row r
    // issued by warp r % 8; the transaction count M * 2K (expected before the
    // wait) stays far below the mbarrier's 2^20 - 1 limit
    const uint32_t sb = smem_u32(&stage_bar);
    if (lane == 0) {
      for (int r = warp; r < M; r += GV_WARPS)
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_u32(ys + r * ys_stride)),
                     "l"(A + int64_t(r) * K), "r"(uint32_t(K) * 2u), "r"(sb)
                     : "memory");
    }
    tc::mbar_wait(sb, 0, 16u);
  }
  if (WTMA) tc::mbar_wait(smem_u32(&w_bar), 0, 16u);
  for (int kb = k0; kb < k1; kb += GV_MAXC * 32) {
    if (WTMA || kb != k0) load_w(kb);
#pragma unroll
    for (int c = 0; c < GV_MAXC; ++c) {
      if (kb + 32 * c >= k1) break;
      const int k = kb + 32 * c + 8 * t;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        const int tok = n * 8 + g;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (tok < M)
          x = (NORM || STAGE) ? *reinterpret_cast<const uint4*>(ys + tok * ys_stride + k)
                              : __ldg(reinterpret_cast<const uint4*>(A + int64_t(tok) * K + k));
#pragma unroll
        for (int tl = 0; tl < TL; ++tl) {
          mma_16816(acc[tl][n], wa[tl][c].x, wb[tl][c].x, wa[tl][c].y, wb[tl][c].y, x.x, x.y);
          mma_16816(acc[tl][n], wa[tl][c].z, wb[tl][c].z, wa[tl][c].w, wb[tl][c].w, x.z, x.w);
        }
      }
    }
  }
  // partial tiles to shared memory: rows 16 tl + g, 16 tl + g + 8; tokens 2t, 2t+1 of each n-tile
#pragma unroll
  for (int tl = 0; tl < TL; ++tl)
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      red[warp][16 * tl + g][n * 8 + 2 * t] = acc[tl][n][0];
      red[warp][16 * tl + g][n * 8 + 2 * t + 1] = acc[tl][n][1];
      red[warp][16 * tl + g + 8][n * 8 + 2 * t] = acc[tl][n][2];
      red[warp][16 * tl + g + 8][n * 8 + 2 * t + 1] = acc[tl][n][3];
    }
  __syncthreads();
  if (EPI == tc::EPI_SILU) {
    for (int e = threadIdx.x; e < 8 * TL * M; e += GV_WARPS * 32) {
      const int r = e & 7, tl = (e >> 3) % TL, tok = (e >> 3) / TL;
      float gs = 0.0f, us = 0.0f;
#pragma unroll
      for (int w = 0; w < GV_WARPS; ++w) {
        gs += red[w][16 * tl + r][tok];
        us += red[w][16 * tl + r + 8][tok];
      }
      const int64_t o = (int64_t(blockIdx.x) * TL + tl) * 8 + r;
      if (o < N / 2) C[int64_t(tok) * ldc + o] = __float2bfloat16_rn(tc::silu_mul_bf16(gs, us));
    }
  } else {
    for (int e = threadIdx.x; e < RPC * TL * M; e += GV_WARPS * 32) {
      const int r = e % (RPC * TL), tok = e / (RPC * TL);
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < GV_WARPS; ++w) sum += red[w][r][tok];   // (RPC == 16 when TL == 2)
      const int64_t row = int64_t(blockIdx.x) * RPC * TL + r;
      if (row < N) C[int64_t(tok) * ldc + row] = __float2bfloat16_rn(sum);
    }
  }
}

// ===========================================================================
// fp32 GEMM on CUDA cores (exact fp32 FMA; the small fp32 model)
// ===========================================================================
__device__ __forceinline__ float w_at(const float* W, int64_t n, int64_t k, int64_t N, int64_t K, int64_t K_l,
                                      int row) {
  if (!row) return W[n * K + k];
  const int64_t r = k / K_l;
  return W[(r * N + n) * K_l + (k - r * K_l)];
}

__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, const float* __restrict__ W,
                                                       float* __restrict__ C, int64_t M, int64_t Nout, int64_t N,
                                                       int64_t K, int64_t K_l, int row, int silu, int64_t i_l) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  __shared__ float sa[16][17];
  __shared__ float sw[2][16][17];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t m = int64_t(blockIdx.y) * 16 + ty;
  const int64_t o = int64_t(blockIdx.x) * 16 + tx;      // output column
  const int64_t o_load = int64_t(blockIdx.x) * 16 + ty; // column whose weights thread (ty, tx) loads
  int64_t n0 = o_load, n1 = 0;
  if (silu) {
    const int64_t r = o_load / i_l, j = o_load % i_l;
    n0 = r * 2 * i_l + j;
    n1 = n0 + i_l;
  }
  float acc0 = 0.0f, acc1 = 0.0f;
  for (int64_t k0 = 0; k0 < K; k0 += 16) {
    const int64_t mm = int64_t(blockIdx.y) * 16 + ty;
    sa[ty][tx] = (mm < M && k0 + tx < K) ? A[mm * K + k0 + tx] : 0.0f;
    const bool ok = o_load < Nout && k0 + tx < K;
    sw[0][ty][tx] = ok ? w_at(W, n0, k0 + tx, N, K, K_l, row) : 0.0f;
    sw[1][ty][tx] = (ok && silu) ? w_at(W, n1, k0 + tx, N, K, K_l, row) : 0.0f;
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      acc0 = fmaf(sa[ty][kk], sw[0][tx][kk], acc0);
      if (silu) acc1 = fmaf(sa[ty][kk], sw[1][tx][kk], acc1);
    }
    __syncthreads();
  }
  if (m < M && o < Nout) {
    float v = acc0;
    if (silu) v = acc0 / (1.0f + expf(-acc0)) * acc1;
    C[m * Nout + o] = v;
  }
}

// ===========================================================================
// host side: tensor maps (cached), planning, launch
// ===========================================================================
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapKey {
  uint64_t ptr;
  uint64_t d[3], s[2];
  uint32_t b[3], rank;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && d[0] == o.d[0] && d[1] == o.d[1] && d[2] == o.d[2] && s[0] == o.s[0] && s[1] == o.s[1] &&
           b[0] == o.b[0] && b[1] == o.b[1] && b[2] == o.b[2] && rank == o.rank;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    for (uint64_t v : {k.d[0], k.d[1], k.d[2], k.s[0], k.s[1], uint64_t(k.b[0]) << 32 | k.b[1],
                       uint64_t(k.b[2]) << 32 | k.rank})
      h = (h ^ v) * 0x100000001B3ull;
    return size_t(h);
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;

}  // namespace

int make_tensor_map(CUtensorMap* out, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box) {
  MapKey key{};
  key.ptr = reinterpret_cast<uint64_t>(ptr);
  key.rank = uint32_t(rank);
  for (int i = 0; i < 3; ++i) {
    key.d[i] = i < rank ? dims[i] : 1;
    key.b[i] = i < rank ? box[i] : 1;
  }
  for (int i = 0; i < 2; ++i) key.s[i] = i < rank - 1 ? strides[i] : 0;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
      *out = it->second;
      return QW_OK;
    }
  }
  auto fn = encode_fn();
  if (!fn) return set_error(QW_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t gd[3] = {key.d[0], key.d[1], key.d[2]};
  cuuint64_t gs[2] = {key.s[0], key.s[1]};
  cuuint32_t bx[3] = {key.b[0], key.b[1], key.b[2]};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), gd, gs, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(QW_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  std::lock_guard<std::mutex> lk(g_map_mu);
  if (g_maps.size() > 8192) g_maps.clear();
  g_maps.emplace(key, *out);
  return QW_OK;
}

namespace {

// 2D (rank 2) or 3D (rank 3) map with box = 64 elements x box_rows (x 1)
int make_map(CUtensorMap* out, const void* ptr, int rank, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s0_bytes,
             uint64_t s1_bytes, uint32_t box_rows) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {s0_bytes, s1_bytes};
  const uint32_t box[3] = {64u, box_rows, 1u};
  return make_tensor_map(out, ptr, rank, dims, strides, box);
}

struct Plan {
  bool swap;
  int bn;
  int splits;         // swap: K-splits per weight tile = cluster size (<= 8)
  int kblocks_total;
  int kpb;
  int p_tiles;        // swap: weight-row tiles (SiluAndMul: 64 gate + 64 up rows per tile)
};

constexpr int kSms = 152;

Plan plan_bf16(int64_t M, int64_t N, int64_t K, int tp, int mode, int epi) {
  Plan p{};
  const int64_t Kl = mode == QW_GEMM_ROW_REDUCE ? K / tp : K;
  p.kpb = int((Kl + tc::BK - 1) / tc::BK);
  p.kblocks_total = mode == QW_GEMM_ROW_REDUCE ? p.kpb * tp : p.kpb;
  p.swap = M <= 64;
  p.splits = 1;
  if (p.swap) {
    p.bn = M <= 16 ? 16 : M <= 32 ? 32 : 64;
    if (epi == QW_EPI_SILU_MUL) {
      const int64_t i_l = N / 2 / tp;
      p.p_tiles = int(tp * ((i_l + tc::BM / 2 - 1) / (tc::BM / 2)));
    } else {
      p.p_tiles = int((N + tc::BM - 1) / tc::BM);
    }
    // about two resident CTAs per SM, at most one cluster of 8 per tile
    int s = (2 * kSms + p.p_tiles - 1) / p.p_tiles;
    s = s < 1 ? 1 : (s > tc::kMaxCluster ? tc::kMaxCluster : s);
    s = s > p.kblocks_total ? p.kblocks_total : s;
    const int per = (p.kblocks_total + s - 1) / s;
    p.splits = (p.kblocks_total + per - 1) / per;
  } else {
    p.bn = 256;
  }
  return p;
}

// args.C as rows of args.ldc bf16 in boxes of 32 rows x 64 columns, the
// epilogue's tensor stores (BoxStore); args.tma_store says whether they apply
// (SiluAndMul: only when no 64-column box crosses a shard's i_l columns)
template <int EPI>
int output_map(CUtensorMap* mC, tc::TcArgs& args) {
  args.tma_store = 0;
  if (EPI == tc::EPI_QKV || args.M <= 0) return QW_OK;
  if (EPI == tc::EPI_SILU && args.i_l % 64 != 0) return QW_OK;
  if ((reinterpret_cast<uintptr_t>(args.C) & 15u) != 0 || (args.ldc * 2) % 16 != 0) return QW_OK;
  const uint64_t dims[2] = {uint64_t(args.ldc), uint64_t(args.M)};
  const uint64_t strides[1] = {uint64_t(args.ldc) * 2};
  const uint32_t box[2] = {64u, 32u};
  const int rc = make_tensor_map(mC, args.C, 2, dims, strides, box);
  if (rc) return rc;
  args.tma_store = 1;
  return QW_OK;
}

template <int BN, int STAGES, bool SWAP, int EPI, bool WROW>
int launch_tc(const CUtensorMap& act, const CUtensorMap& w, const tc::TcArgs& args_in, int splits, cudaStream_t st) {
  auto kern = tc::gemm_tc_kernel<BN, STAGES, SWAP, EPI, WROW>;
  tc::TcArgs args = args_in;
  CUtensorMap mC = act;   // (unused unless args.tma_store)
  args.tma_store = 0;
  // tensor-store epilogue for plain outputs (measured: QKV 134 -> 122 us, o_proj
  // 71 -> 68 us, down 95 -> 93 us for 8 x 2048 tokens; the SiluAndMul tile
  // stores directly: 211 us against 303 us with tensor stores)
  if (!SWAP && splits == 1 && EPI == tc::EPI_NONE) {
    const int rc = output_map<EPI>(&mC, args);
    if (rc) return rc;
  }
  constexpr size_t smem = tc::smem_bytes<BN, STAGES>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(args.p_tiles * args.q_tiles), unsigned(splits), 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = unsigned(splits);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, act, w, mC, args);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemm_tc_kernel launch: %s", cudaGetErrorString(e));
  return check_launch("gemm_tc_kernel");
}

template <int EPI, bool WROW>
int launch_tc_m256(const CUtensorMap& act, const CUtensorMap& w, const tc::TcArgs& args_in, cudaStream_t st) {
  auto kern = tc::gemm_tc_m256_kernel<EPI, WROW>;
  constexpr size_t smem = tc::m2_smem_bytes();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  tc::TcArgs args = args_in;
  CUtensorMap mC = act;   // (unused unless args.tma_store)
  args.tma_store = 0;
  if (EPI == tc::EPI_NONE) {
    const int rc = output_map<EPI>(&mC, args);
    if (rc) return rc;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(args.p_tiles * args.q_tiles), 1, 1);
  cfg.blockDim = dim3(tc::M2_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.numAttrs = 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, act, w, mC, args);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemm_tc_m256_kernel launch: %s", cudaGetErrorString(e));
  return check_launch("gemm_tc_m256_kernel");
}

static int gv_device_sms();

// The persistent prefill GEMM (gemm_tc_persist_kernel) replaces the one-tile-
// per-CTA kernel for many-token GEMMs while QW_TC_PERSISTENT=1 (read at each
// call: one process can compare both).
bool tc_persistent_enabled() {
  const char* v = getenv("QW_TC_PERSISTENT");
  return v && v[0] == '1';
}

template <int EPI, bool WROW>
int launch_tc_persist(const CUtensorMap& act, const CUtensorMap& w, const tc::TcArgs& args_in, cudaStream_t st) {
  auto kern = tc::gemm_tc_persist_kernel<EPI, WROW>;
  constexpr size_t smem = tc::psmem_bytes();
  tc::TcArgs args = args_in;
  CUtensorMap mC = act;   // (unused unless args.tma_store)
  {
    const int rc = output_map<EPI>(&mC, args);
    if (rc) return rc;
  }
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  // one CTA per SM (the ring takes the shared memory, the two accumulators all of TMEM)
  const int64_t n_tiles = int64_t(args.p_tiles) * args.q_tiles;
  const int64_t grid = n_tiles < gv_device_sms() ? n_tiles : gv_device_sms();
  if (grid <= 0) return QW_OK;
  if (n_tiles > INT32_MAX || ((n_tiles + grid - 1) / grid) * int64_t(args.kblocks_total) > INT32_MAX)
    return set_error(QW_ERR_SHAPE, "gemm_tc_persist_kernel: too many tiles");
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid), 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.numAttrs = 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, act, w, mC, args);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemm_tc_persist_kernel launch: %s", cudaGetErrorString(e));
  return check_launch("gemm_tc_persist_kernel");
}

// Lets kernel `kern` take `smem` bytes of dynamic shared memory: the default
// allows 48 KB minus its static shared memory; beyond that it opts in (once
// per size growth).  `allowed` is the caller's per-kernel record.
static int gv_allow_smem(const void* kern, size_t smem, size_t& allowed) {
  if (allowed == 0) {
    cudaFuncAttributes fa;
    const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
    allowed = 48 * 1024 - fa.sharedSizeBytes;
  }
  if (smem > allowed) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    allowed = smem;
  }
  return QW_OK;
}

int gemm_bf16(const bf16* A, const bf16* W, bf16* C, int64_t M, int64_t N, int64_t K, int tp, int mode, int epi,
              cudaStream_t st) {
  const Plan p = plan_bf16(M, N, K, tp, mode, epi);
  const int64_t Kl = mode == QW_GEMM_ROW_REDUCE ? K / tp : K;
  const bool wrow = mode == QW_GEMM_ROW_REDUCE;
  int rc;
  CUtensorMap mA, mW;
  tc::TcArgs a{};
  a.C = C;
  a.ldc = epi == QW_EPI_SILU_MUL ? N / 2 : N;
  a.M = M;
  a.N = N;
  a.kblocks_total = p.kblocks_total;
  a.kpb = p.kpb;
  a.k_shard = Kl;
  a.i_l = epi == QW_EPI_SILU_MUL ? N / 2 / tp : 0;
  a.splits = 1;
  if (!p.swap) {
    rc = make_map(&mA, A, 2, uint64_t(K), uint64_t(M), 1, uint64_t(K) * 2, 0, tc::BM);
    if (rc) return rc;
    a.p_tiles = int((M + tc::BM - 1) / tc::BM);
    if (epi == QW_EPI_SILU_MUL) {
      a.silu_tps = int((a.i_l + p.bn / 2 - 1) / (p.bn / 2));
      a.q_tiles = a.silu_tps * tp;
    } else {
      a.q_tiles = int((N + p.bn - 1) / p.bn);
    }
    const bool persistent = tc_persistent_enabled();
    const uint32_t wrows = epi == QW_EPI_SILU_MUL ? uint32_t(p.bn / 2) : uint32_t(p.bn);
    if (wrow) rc = make_map(&mW, W, 3, uint64_t(Kl), uint64_t(N), uint64_t(tp), uint64_t(Kl) * 2,
                            uint64_t(Kl) * 2 * uint64_t(N), wrows);
    else rc = make_map(&mW, W, 2, uint64_t(K), uint64_t(N), 1, uint64_t(K) * 2, 0, wrows);
    if (rc) return rc;
    a.p_fastest = (M * K * 2) <= (int64_t(48) << 20) ? 1 : 0;
    a.kblocks = p.kblocks_total;
    if (persistent) {
      if (epi == QW_EPI_SILU_MUL) return launch_tc_persist<tc::EPI_SILU, false>(mA, mW, a, st);
      if (wrow) return launch_tc_persist<tc::EPI_NONE, true>(mA, mW, a, st);
      return launch_tc_persist<tc::EPI_NONE, false>(mA, mW, a, st);
    }
    // 256-row tiles while they still fill every SM at least once
    const int64_t p256 = (M + tc::M2_ROWS - 1) / tc::M2_ROWS;
    if (p256 * a.q_tiles >= gv_device_sms()) {
      rc = make_map(&mA, A, 2, uint64_t(K), uint64_t(M), 1, uint64_t(K) * 2, 0, uint32_t(tc::M2_ROWS));
      if (rc) return rc;
      a.p_tiles = int(p256);
      if (epi == QW_EPI_SILU_MUL) return launch_tc_m256<tc::EPI_SILU, false>(mA, mW, a, st);
      if (wrow) return launch_tc_m256<tc::EPI_NONE, true>(mA, mW, a, st);
      return launch_tc_m256<tc::EPI_NONE, false>(mA, mW, a, st);
    }
    if (epi == QW_EPI_SILU_MUL) return launch_tc<256, 4, false, tc::EPI_SILU, false>(mA, mW, a, 1, st);
    if (wrow) return launch_tc<256, 4, false, tc::EPI_NONE, true>(mA, mW, a, 1, st);
    return launch_tc<256, 4, false, tc::EPI_NONE, false>(mA, mW, a, 1, st);
  }
  // few tokens, moderate N: weight streaming on warp-level MMA (see gemv_mma_kernel)
  if (p.splits > 1 && Kl % 32 == 0) {
    const int nt = M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8;
    const bool small_k = K <= GV_WARPS * 32 * 4;            // every warp's weights fit 4 chunks
    // up to 8 tokens: activations staged in shared memory (measured on the
    // 28-layer decode step, 128 steps: 139.3 -> 136.3 ms with per-thread
    // asynchronous copies, 134.2 -> 125.1 ms on moving to one bulk copy per row)
    const size_t stage_smem = size_t(M) * (K + GV_YPAD) * 2;
    const bool stage = M <= 8 && stage_smem <= size_t(200) * 1024;
    // 8 rows per CTA (twice the CTAs) for narrow outputs, except on the staged
    // path: every CTA there copies all the activation rows, and 16 rows per CTA
    // halve that traffic (decode o_proj / down: 118.0 -> 116.0 ms per 128 steps
    // together with the two-tile QKV GEMV)
    const bool half = epi != QW_EPI_SILU_MUL && N <= 2048 && !(nt == 1 && stage);
    const unsigned blocks =
        unsigned(epi == QW_EPI_SILU_MUL ? (N / 2 + 7) / 8 : half ? (N + 7) / 8 : (N + 15) / 16);
    cudaError_t e;
  // and the weight rows bulk-copied into shared memory beside them (WTMA)
#define QW_GV_ONE(NTV, EPIV, WR, RPCV, MC)                                                                     \
  if (NTV == 1 && stage) {                                                                                     \
    const size_t wsm_ = size_t(EPIV == tc::EPI_SILU || RPCV == 16 ? 16 : 8) * (K + gv_wpad(int(K))) * 2;       \
    const NormArgs na_{nullptr, nullptr, nullptr, 0.0f};                                                       \
    if (stage_smem + wsm_ <= size_t(200) * 1024) {                                                             \
      auto kern = gemv_mma_kernel<1, EPIV, WR, RPCV, 4, false, 1, true, true>;                                 \
      static size_t allowed = 0;                                                                               \
      const int rc_ = gv_allow_smem(reinterpret_cast<const void*>(kern), stage_smem + wsm_, allowed);         \
      if (rc_) return rc_;                                                                                     \
      e = launch_pdl(kern, dim3(blocks), dim3(GV_WARPS * 32), stage_smem + wsm_, st, A, W, C, int(M), int(N),  \
                     int(K), int(Kl), a.ldc, a.i_l, na_);                                                      \
    } else {                                                                                                   \
      auto kern = gemv_mma_kernel<1, EPIV, WR, RPCV, MC, false, 1, true>;                                      \
      static size_t allowed = 0;                                                                               \
      const int rc_ = gv_allow_smem(reinterpret_cast<const void*>(kern), stage_smem, allowed);                \
      if (rc_) return rc_;                                                                                     \
      e = launch_pdl(kern, dim3(blocks), dim3(GV_WARPS * 32), stage_smem, st, A, W, C, int(M), int(N), int(K), \
                     int(Kl), a.ldc, a.i_l, na_);                                                              \
    }                                                                                                          \
  } else {                                                                                                     \
    e = launch_pdl(gemv_mma_kernel<NTV, EPIV, WR, RPCV, MC>, dim3(blocks), dim3(GV_WARPS * 32), 0, st, A, W, C, \
                   int(M), int(N), int(K), int(Kl), a.ldc, a.i_l, NormArgs{nullptr, nullptr, nullptr, 0.0f}); \
  }
#define QW_GV(NTV)                                                                                             \
  if (epi == QW_EPI_SILU_MUL) {                                                                                \
    if (small_k) { QW_GV_ONE(NTV, tc::EPI_SILU, false, 16, 4) } else { QW_GV_ONE(NTV, tc::EPI_SILU, false, 16, 12) } \
  } else if (half) {                                                                                           \
    if (wrow) { QW_GV_ONE(NTV, tc::EPI_NONE, true, 8, 12) } else { QW_GV_ONE(NTV, tc::EPI_NONE, false, 8, 12) } \
  } else if (small_k) {                                                                                        \
    if (wrow) { QW_GV_ONE(NTV, tc::EPI_NONE, true, 16, 4) } else { QW_GV_ONE(NTV, tc::EPI_NONE, false, 16, 4) } \
  } else {                                                                                                     \
    if (wrow) { QW_GV_ONE(NTV, tc::EPI_NONE, true, 16, 12) } else { QW_GV_ONE(NTV, tc::EPI_NONE, false, 16, 12) } \
  }
    if (nt == 1) { QW_GV(1) }
    else if (nt == 2) { QW_GV(2) }
    else if (nt == 4) { QW_GV(4) }
    else { QW_GV(8) }
#undef QW_GV
#undef QW_GV_ONE
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemv_mma_kernel launch: %s", cudaGetErrorString(e));
    return check_launch("gemv_mma_kernel");
  }
  // swapped operands for few tokens
  rc = make_map(&mA, A, 2, uint64_t(K), uint64_t(M), 1, uint64_t(K) * 2, 0, uint32_t(p.bn));
  if (rc) return rc;
  const uint32_t wrows = epi == QW_EPI_SILU_MUL ? uint32_t(tc::BM / 2) : uint32_t(tc::BM);
  if (wrow) rc = make_map(&mW, W, 3, uint64_t(Kl), uint64_t(N), uint64_t(tp), uint64_t(Kl) * 2,
                          uint64_t(Kl) * 2 * uint64_t(N), wrows);
  else rc = make_map(&mW, W, 2, uint64_t(K), uint64_t(N), 1, uint64_t(K) * 2, 0, wrows);
  if (rc) return rc;
  a.p_tiles = p.p_tiles;
  a.q_tiles = 1;
  a.p_fastest = 1;
  a.kblocks = (p.kblocks_total + p.splits - 1) / p.splits;
  a.splits = p.splits;
  if (epi == QW_EPI_SILU_MUL) a.silu_tps = p.p_tiles / tp;
#define QW_SWAP_LAUNCH(BNV)                                                                                \
  if (epi == QW_EPI_SILU_MUL) return launch_tc<BNV, 4, true, tc::EPI_SILU, false>(mA, mW, a, p.splits, st); \
  if (wrow) return launch_tc<BNV, 4, true, tc::EPI_NONE, true>(mA, mW, a, p.splits, st);                    \
  return launch_tc<BNV, 4, true, tc::EPI_NONE, false>(mA, mW, a, p.splits, st);
  if (p.bn == 16) { QW_SWAP_LAUNCH(16) }
  if (p.bn == 32) { QW_SWAP_LAUNCH(32) }
  QW_SWAP_LAUNCH(64)
#undef QW_SWAP_LAUNCH
}

// y = RMSNorm(x + res_in) * gamma (in every CTA's shared memory), C = y W^T,
// for at most 16 tokens: the weight-streaming GEMV with a norm prologue.
// SMs of the current device (152 when it cannot be queried)
static int gv_device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

int norm_gemm_bf16(const bf16* x, const NormArgs& na, const bf16* W, bf16* C, int M, int N, int K, int tp, int epi,
                   cudaStream_t st) {
  const int nt = M <= 8 ? 1 : 2;
  const bool small_k = K <= GV_WARPS * 32 * 4;
  const bool half = epi != QW_EPI_SILU_MUL && N <= 2048;
  unsigned blocks = unsigned(epi == QW_EPI_SILU_MUL ? (N / 2 + 7) / 8 : half ? (N + 7) / 8 : (N + 15) / 16);
  // SiluAndMul with more 8-output CTAs than fit at once (two per SM): 16 outputs
  // per CTA, so the norm prologue is not repeated by a second wave.  Plain
  // outputs with more 16-row CTAs than SMs: 32 rows per CTA (decode QKV: with
  // the 16-row staged GEMVs, 118.0 -> 116.0 ms per 128 steps)
  const bool two_tiles = small_k && !half && (epi == QW_EPI_SILU_MUL || nt == 1) &&
                         blocks > unsigned((epi == QW_EPI_SILU_MUL ? 2 : 1) * gv_device_sms());
  if (two_tiles) blocks = (blocks + 1) / 2;
  const int64_t ldc = epi == QW_EPI_SILU_MUL ? N / 2 : N;
  const int64_t i_l = epi == QW_EPI_SILU_MUL ? N / 2 / tp : 0;
  const size_t smem = size_t(M) * (K + GV_YPAD) * 2;
  cudaError_t e = cudaSuccess;
#define QW_NG_ONE(NTV, EPIV, RPCV, MC, TLV)                                                                      \
  {                                                                                                              \
    const size_t wsm_ = size_t(EPIV == tc::EPI_SILU || RPCV == 16 ? 16 : 8) * TLV * (K + gv_wpad(K)) * 2;        \
    if (NTV == 1 && smem + wsm_ <= size_t(200) * 1024) {   /* weight rows bulk-copied into shared memory */      \
      auto kern = gemv_mma_kernel<1, EPIV, false, RPCV, 4, true, TLV, false, true>;                              \
      static size_t allowed = 0;                                                                                 \
      const int rc_ = gv_allow_smem(reinterpret_cast<const void*>(kern), smem + wsm_, allowed);                 \
      if (rc_) return rc_;                                                                                       \
      e = launch_pdl(kern, dim3(blocks), dim3(GV_WARPS * 32), smem + wsm_, st, x, W, C, M, N, K, K, ldc, i_l,    \
                     na);                                                                                        \
    } else {                                                                                                     \
      auto kern = gemv_mma_kernel<NTV, EPIV, false, RPCV, MC, true, TLV>;                                        \
      static size_t allowed = 0;                                                                                 \
      const int rc_ = gv_allow_smem(reinterpret_cast<const void*>(kern), smem, allowed);                        \
      if (rc_) return rc_;                                                                                       \
      e = launch_pdl(kern, dim3(blocks), dim3(GV_WARPS * 32), smem, st, x, W, C, M, N, K, K, ldc, i_l, na);      \
    }                                                                                                            \
  }
#define QW_NG(NTV)                                                                                               \
  if (epi == QW_EPI_SILU_MUL) {                                                                                  \
    if (two_tiles) QW_NG_ONE(NTV, tc::EPI_SILU, 16, 4, 2)                                                        \
    else if (small_k) QW_NG_ONE(NTV, tc::EPI_SILU, 16, 4, 1)                                                     \
    else QW_NG_ONE(NTV, tc::EPI_SILU, 16, 12, 1)                                                                 \
  } else if (half) {                                                                                             \
    QW_NG_ONE(NTV, tc::EPI_NONE, 8, 12, 1)                                                                       \
  } else if (small_k) {                                                                                          \
    if (two_tiles) QW_NG_ONE(NTV, tc::EPI_NONE, 16, 4, 2)                                                        \
    else QW_NG_ONE(NTV, tc::EPI_NONE, 16, 4, 1)                                                                  \
  } else {                                                                                                       \
    QW_NG_ONE(NTV, tc::EPI_NONE, 16, 12, 1)                                                                      \
  }
  if (nt == 1) { QW_NG(1) } else { QW_NG(2) }
#undef QW_NG
#undef QW_NG_ONE
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemv_mma_kernel launch: %s", cudaGetErrorString(e));
  return check_launch("gemv_mma_kernel (norm prologue)");
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

unsigned int take_tc_timeouts() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, tc::g_tc_timeout, sizeof(v));
  if (v) cudaMemcpyToSymbol(tc::g_tc_timeout, &z, sizeof(z));
  return v;
}

}  // namespace qw

using namespace qw;

static int gemm_check(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K, int tp, int mode,
                      int epi, int dtype, const char* who) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "%s: dtype %d", who, dtype);
  if (M < 0 || N <= 0 || K <= 0 || tp <= 0) return set_error(QW_ERR_INVALID_ARG, "%s: bad sizes", who);
  if (mode != QW_GEMM_COLUMN && mode != QW_GEMM_ROW_REDUCE)
    return set_error(QW_ERR_INVALID_ARG, "%s: mode %d", who, mode);
  if (epi != QW_EPI_NONE && epi != QW_EPI_SILU_MUL) return set_error(QW_ERR_INVALID_ARG, "%s: epilogue %d", who, epi);
  if (epi == QW_EPI_SILU_MUL && mode != QW_GEMM_COLUMN)
    return set_error(QW_ERR_INVALID_ARG, "%s: SiluAndMul needs the column (gate_up) layout", who);
  if (mode == QW_GEMM_ROW_REDUCE && K % tp) return set_error(QW_ERR_SHAPE, "%s: K=%lld %% tp=%d", who, (long long)K, tp);
  if (mode == QW_GEMM_COLUMN && N % tp) return set_error(QW_ERR_SHAPE, "%s: N=%lld %% tp=%d", who, (long long)N, tp);
  if (epi == QW_EPI_SILU_MUL && (N % (2 * tp)))
    return set_error(QW_ERR_SHAPE, "%s: gate_up width %lld not 2*tp*I_l", who, (long long)N);
  if (M == 0) return QW_OK;
  if (!A || !W || !C) return set_error(QW_ERR_INVALID_ARG, "%s: null pointer", who);
  if (dtype == QW_BF16) {
    const int64_t Kl = mode == QW_GEMM_ROW_REDUCE ? K / tp : K;
    if (K % 8 || Kl % 8) return set_error(QW_ERR_SHAPE, "%s: K and K/tp must be multiples of 8", who);
    if (N % 16) return set_error(QW_ERR_SHAPE, "%s: N must be a multiple of 16", who);
    if (epi == QW_EPI_SILU_MUL && ((N / 2 / tp) % 8))
      return set_error(QW_ERR_SHAPE, "%s: I/tp must be a multiple of 8", who);
    if (!al16(A) || !al16(W) || !al16(C)) return set_error(QW_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
    if (N > (int64_t(1) << 31) || M > (int64_t(1) << 31) || K > (int64_t(1) << 31))
      return set_error(QW_ERR_SHAPE, "%s: dimension too large", who);
  }
  return -1;  // continue
}

extern "C" size_t qw_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int tp, int mode, int epilogue, int dtype) {
  (void)M, (void)N, (void)K, (void)tp, (void)mode, (void)epilogue, (void)dtype;
  return 0;   // split-K partials stay on chip (cluster shared memory)
}

extern "C" int qw_gemm(const void* A, const void* W, void* C, int64_t M, int64_t N, int64_t K, int tp, int mode,
                       int epilogue, void* workspace, size_t workspace_bytes, int dtype, void* stream) {
  (void)workspace, (void)workspace_bytes;
  int rc = gemm_check(A, W, C, M, N, K, tp, mode, epilogue, dtype, "qw_gemm");
  if (rc >= 0) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == QW_F32) {
    const int64_t Nout = epilogue == QW_EPI_SILU_MUL ? N / 2 : N;
    const int64_t Kl = mode == QW_GEMM_ROW_REDUCE ? K / tp : K;
    dim3 grid(unsigned((Nout + 15) / 16), unsigned((M + 15) / 16));
    launch_pdl(gemm_f32_kernel, grid, 256, 0, st, static_cast<const float*>(A), static_cast<const float*>(W),
                                          static_cast<float*>(C), M, Nout, N, K, Kl, mode == QW_GEMM_ROW_REDUCE,
                                          epilogue == QW_EPI_SILU_MUL, epilogue == QW_EPI_SILU_MUL ? N / 2 / tp : 0);
    return check_launch("gemm_f32_kernel");
  }
  return gemm_bf16(static_cast<const bf16*>(A), static_cast<const bf16*>(W), static_cast<bf16*>(C), M, N, K, tp,
                   mode, epilogue, st);
}

static size_t lm_rows_bytes(int64_t n_out, int64_t H, int dtype) {
  const size_t es = dtype == QW_BF16 ? 2 : 4;
  return (size_t(n_out) * size_t(H) * es + 255) / 256 * 256;
}

extern "C" size_t qw_lm_head_workspace_size(int64_t n_out, int64_t V, int64_t H, int tp, int dtype) {
  if (n_out <= 0 || V <= 0 || H <= 0) return 0;
  (void)tp;
  return kCounterBytes + lm_rows_bytes(n_out, H, dtype);
}

extern "C" int qw_lm_head(const void* hidden, int64_t T, const int32_t* last_idx, int64_t n_out, const void* table,
                          int64_t V, int64_t H, int tp, void* logits, int64_t* next_tokens, void* workspace,
                          size_t workspace_bytes, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_lm_head: dtype %d", dtype);
  if (T < 0 || n_out < 0 || V <= 0 || H <= 0 || tp <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_lm_head: bad sizes");
  if (V % tp) return set_error(QW_ERR_SHAPE, "qw_lm_head: V=%lld %% tp=%d", (long long)V, tp);
  if (n_out == 0) return QW_OK;
  if (!hidden || !table || !logits) return set_error(QW_ERR_INVALID_ARG, "qw_lm_head: null pointer");
  if (!last_idx && n_out > T) return set_error(QW_ERR_SHAPE, "qw_lm_head: n_out > T without last_idx");
  const size_t es = dtype == QW_BF16 ? 2 : 4;
  int rc = gemm_check(hidden, table, logits, n_out, V, H, 1, QW_GEMM_COLUMN, QW_EPI_NONE, dtype, "qw_lm_head");
  if (rc >= 0) return rc;
  if ((H * int64_t(es)) % 16 || !al16(hidden)) return set_error(QW_ERR_INVALID_ARG, "qw_lm_head: H rows must be 16-byte");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* x = hidden;
  if (last_idx) {
    const size_t need = qw_lm_head_workspace_size(n_out, V, H, tp, dtype);
    if (!workspace || workspace_bytes < need)
      return set_error(QW_ERR_WORKSPACE, "qw_lm_head: workspace of %zu bytes needed", need);
    // the selected rows go after the counter area that other calls may share
    uint8_t* rows = static_cast<uint8_t*>(workspace) + kCounterBytes;
    rc = dtype == QW_BF16 ? launch_gather_rows<bf16>(hidden, T, last_idx, n_out, H, rows, st)
                          : launch_gather_rows<float>(hidden, T, last_idx, n_out, H, rows, st);
    if (rc) return rc;
    x = rows;
  }
  // each vocab shard r projects onto its rows [r*V/tp, (r+1)*V/tp) and writes
  // logit columns [r*V/tp, (r+1)*V/tp): with the shards stacked in one table
  // that is a single column-split GEMM over the whole vocab
  rc = qw_gemm(x, table, logits, n_out, V, H, 1, QW_GEMM_COLUMN, QW_EPI_NONE, nullptr, 0, dtype, stream);
  if (rc) return rc;
  if (next_tokens) return qw_argmax(logits, n_out, V, next_tokens, dtype, stream);
  return QW_OK;
}

extern "C" int qw_add_rmsnorm_gemm(const void* x, const void* residual_in, void* residual_out, const void* gamma,
                                   float eps, const void* W, void* C, int64_t M, int64_t N, int64_t K, int tp,
                                   int epilogue, int dtype, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_add_rmsnorm_gemm: bf16 only");
  if (M < 0 || M > 16 || N <= 0 || K <= 0 || tp <= 0)
    return set_error(QW_ERR_SHAPE, "qw_add_rmsnorm_gemm: needs 0 <= M <= 16 tokens");
  if (epilogue != QW_EPI_NONE && epilogue != QW_EPI_SILU_MUL)
    return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm_gemm: epilogue %d", epilogue);
  if (K % 32 || N % 16 || N % tp || (epilogue == QW_EPI_SILU_MUL && ((N % (2 * tp)) || (N / 2 / tp) % 8)))
    return set_error(QW_ERR_SHAPE, "qw_add_rmsnorm_gemm: K %% 32, N %% 16 and the gate_up split rules");
  // the normed rows of all tokens sit in shared memory beside the <= 16 KB reduction tile
  if (size_t(M) * (K + GV_YPAD) * 2 > size_t(211) * 1024)
    return set_error(QW_ERR_SHAPE, "qw_add_rmsnorm_gemm: %lld tokens x K %lld exceed shared memory",
                     (long long)M, (long long)K);
  if (M == 0) return QW_OK;
  if (!x || !gamma || !W || !C) return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm_gemm: null pointer");
  if (!al16(x) || !al16(W) || !al16(C) || !al16(gamma) || (residual_in && !al16(residual_in)) ||
      (residual_out && !al16(residual_out)))
    return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm_gemm: pointers must be 16-byte aligned");
  if (residual_out != nullptr && (residual_out == x || residual_out == residual_in))
    return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm_gemm: residual_out must not alias x or residual_in");
  const NormArgs na{static_cast<const bf16*>(residual_in), static_cast<bf16*>(residual_out),
                    static_cast<const bf16*>(gamma), eps};
  return norm_gemm_bf16(static_cast<const bf16*>(x), na, static_cast<const bf16*>(W), static_cast<bf16*>(C), int(M),
                        int(N), int(K), tp, epilogue, static_cast<cudaStream_t>(stream));
}

// A row-parallel Linear (o_proj, down_proj) whose output joins the residual
// stream, followed by the next RMSNorm ([SK] §1-§2 add_rms_forward, [TP] §3):
// the tcgen05 GEMM of many tokens with an epilogue that adds the residual and
// normalises the row.  The N / 256 tiles of a 128-row block form one thread-
// block cluster and exchange their rows' sums of squares over distributed
// shared memory.
extern "C" int qw_gemm_add_rmsnorm(const void* A, const void* W, int64_t M, int64_t N, int64_t K, int tp,
                                   void* residual, const void* gamma, float eps, void* y, int dtype, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_gemm_add_rmsnorm: bf16 only");
  if (M < 0 || N <= 0 || K <= 0 || tp <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_gemm_add_rmsnorm: bad sizes");
  if (N % 256 || N / 256 > tc::kMaxCluster || K % tp || (K / tp) % 8)
    return set_error(QW_ERR_SHAPE, "qw_gemm_add_rmsnorm: needs N a multiple of 256 up to 2048 and K/tp %% 8 == 0");
  if (M == 0) return QW_OK;
  if (!A || !W || !residual || !gamma || !y) return set_error(QW_ERR_INVALID_ARG, "qw_gemm_add_rmsnorm: null pointer");
  const uintptr_t al = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(W) |
                       reinterpret_cast<uintptr_t>(residual) | reinterpret_cast<uintptr_t>(gamma) |
                       reinterpret_cast<uintptr_t>(y);
  if (al % 16) return set_error(QW_ERR_INVALID_ARG, "qw_gemm_add_rmsnorm: pointers must be 16-byte aligned");
  if (y == residual) return set_error(QW_ERR_INVALID_ARG, "qw_gemm_add_rmsnorm: y must not alias the residual");
  const int64_t Kl = K / tp;
  const int kpb = int((Kl + tc::BK - 1) / tc::BK);
  CUtensorMap mA, mW;
  int rc = make_map(&mA, A, 2, uint64_t(K), uint64_t(M), 1, uint64_t(K) * 2, 0, tc::BM);
  if (rc) return rc;
  rc = make_map(&mW, W, 3, uint64_t(Kl), uint64_t(N), uint64_t(tp), uint64_t(Kl) * 2, uint64_t(Kl) * 2 * uint64_t(N),
                256u);
  if (rc) return rc;
  tc::TcArgs a{};
  a.C = nullptr;
  a.ldc = N;
  a.M = M;
  a.N = N;
  a.kpb = kpb;
  a.kblocks_total = kpb * tp;
  a.kblocks = kpb * tp;
  a.k_shard = Kl;
  a.splits = 1;
  a.p_tiles = int((M + tc::BM - 1) / tc::BM);
  a.q_tiles = int(N / 256);
  a.p_fastest = 0;   // the tiles of one row block are consecutive: one cluster
  a.eps = eps;
  a.resid = static_cast<bf16*>(residual);
  a.y_out = static_cast<bf16*>(y);
  a.norm_gamma = static_cast<const bf16*>(gamma);
  // 256-row tiles while they still fill every SM at least once
  const int64_t p256 = (M + tc::M2_ROWS - 1) / tc::M2_ROWS;
  const bool m256 = p256 * a.q_tiles >= gv_device_sms();
  if (m256) {
    rc = make_map(&mA, A, 2, uint64_t(K), uint64_t(M), 1, uint64_t(K) * 2, 0, uint32_t(tc::M2_ROWS));
    if (rc) return rc;
    a.p_tiles = int(p256);
  }
  auto kern = m256 ? tc::gemm_tc_m256_kernel<tc::EPI_ADDNORM, true> : tc::gemm_tc_kernel<256, 4, false, tc::EPI_ADDNORM, true>;
  const size_t smem = m256 ? tc::m2_smem_bytes() : tc::smem_bytes<256, 4>();
  static bool configured[2] = {false, false};
  if (!configured[m256]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured[m256] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(a.p_tiles * a.q_tiles), 1, 1);
  cfg.blockDim = dim3(m256 ? tc::M2_THREADS : 192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(a.q_tiles);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  a.tma_store = 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, mA, mW, mA, a);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "gemm_tc_kernel (add + RMSNorm) launch: %s", cudaGetErrorString(e));
  return check_launch("gemm_tc_kernel (add + RMSNorm)");
}

// The merged QKV projection of many tokens with its QK-RMSNorm + RoPE + KV
// store as the tcgen05 GEMM's epilogue (prefill): the QKV output never goes
// to memory.  Same results, bit for bit, as qw_gemm (COLUMN) followed by
// qw_qkv_norm_rope_store_kv.
extern "C" int qw_qkv_gemm_norm_rope_store_kv(const void* A, const void* W, int64_t T, int64_t H, int n_heads,
                                              int n_kv_heads, int head_dim, int tp, const int64_t* positions,
                                              const float* cos_sin, int64_t max_position, const void* q_gamma,
                                              const void* k_gamma, float eps, const int64_t* slot_mapping,
                                              void* k_cache, void* v_cache, int64_t num_slots, void* q_out,
                                              int32_t* err_count, int dtype, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_qkv_gemm_norm_rope_store_kv: bf16 only");
  if (T < 0 || H <= 0 || n_heads <= 0 || n_kv_heads <= 0 || tp <= 0 || max_position <= 0 || num_slots < 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_qkv_gemm_norm_rope_store_kv: bad sizes");
  if (head_dim != 128 || n_heads % tp || n_kv_heads % tp || ((n_heads + 2 * n_kv_heads) / tp) % 2 || H % 8)
    return set_error(QW_ERR_SHAPE,
                     "qw_qkv_gemm_norm_rope_store_kv: needs head_dim 128, tp | nh and nkv, an even number of heads "
                     "per shard and H %% 8 == 0");
  if (T == 0) return QW_OK;
  if (!A || !W || !positions || !cos_sin || !q_gamma || !k_gamma || !slot_mapping || !k_cache || !v_cache || !q_out)
    return set_error(QW_ERR_INVALID_ARG, "qw_qkv_gemm_norm_rope_store_kv: null pointer");
  const uintptr_t al = reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(W) |
                       reinterpret_cast<uintptr_t>(cos_sin) | reinterpret_cast<uintptr_t>(q_gamma) |
                       reinterpret_cast<uintptr_t>(k_gamma) | reinterpret_cast<uintptr_t>(k_cache) |
                       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(q_out);
  if (al % 16) return set_error(QW_ERR_INVALID_ARG, "qw_qkv_gemm_norm_rope_store_kv: pointers must be 16-byte aligned");
  const int64_t N = int64_t(n_heads + 2 * n_kv_heads) * 128;
  const int kblocks = int((H + tc::BK - 1) / tc::BK);   // one 128 x 256 tile per CTA over the whole K
  CUtensorMap mA, mW;
  int rc = make_map(&mA, A, 2, uint64_t(H), uint64_t(T), 1, uint64_t(H) * 2, 0, tc::BM);
  if (rc) return rc;
  rc = make_map(&mW, W, 2, uint64_t(H), uint64_t(N), 1, uint64_t(H) * 2, 0, 256u);
  if (rc) return rc;
  tc::TcArgs a{};
  a.C = nullptr;
  a.ldc = N;
  a.M = T;
  a.N = N;
  a.kblocks_total = kblocks;
  a.kpb = kblocks;
  a.k_shard = H;
  a.splits = 1;
  a.p_tiles = int((T + tc::BM - 1) / tc::BM);
  a.q_tiles = int(N / 256);
  a.p_fastest = (T * H * 2) <= (int64_t(48) << 20) ? 1 : 0;
  a.kblocks = kblocks;
  a.positions = positions;
  a.cos_sin = cos_sin;
  a.max_pos = max_position;
  a.q_gamma = static_cast<const bf16*>(q_gamma);
  a.k_gamma = static_cast<const bf16*>(k_gamma);
  a.eps = eps;
  a.slots = slot_mapping;
  a.k_cache = static_cast<bf16*>(k_cache);
  a.v_cache = static_cast<bf16*>(v_cache);
  a.num_slots = num_slots;
  a.q_out = static_cast<bf16*>(q_out);
  a.err = err_count;
  a.nh = n_heads;
  a.nkv = n_kv_heads;
  a.tp = tp;
  // persistent: one CTA per SM, two TMEM accumulators, so each tile's longer
  // epilogue runs while the MMAs of the CTA's next tile proceed
  // (on the persistent kernel, where the epilogue overlaps the next tile's
  // mainloop; a one-tile 256-row version measured slower: 20.5 against 19.6 ms
  // for the 8 x 2048 prefill)
  return launch_tc_persist<tc::EPI_QKV, false>(mA, mW, a, static_cast<cudaStream_t>(stream));
}

extern "C" int qw_selftest_wait_timeout(void* stream) {
  tc::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  return check_launch("qw_selftest_wait_timeout");
}
