// Memory-bound steps of the Qwen3 forward pass: vocab-parallel embedding,
// fused residual add + RMSNorm, QK-RMSNorm + RoPE + KV-cache store,
// SiluAndMul, greedy argmax and the last-token row gather.
//
// All of them move each byte once with 16-byte coalesced accesses and reduce
// with warp shuffles; their roofline is HBM bandwidth.
#include <math.h>

#include "common.cuh"

namespace qw {

// ===========================================================================
// vocab-parallel embedding  ([VH] §3 five steps, [VPE], [SK] §6)
// one warp per token; the per-shard mask/shift/gather/zero/sum is evaluated
// for every shard, and only the owning shard's row is read.
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(256) embed_vocab_kernel(const int64_t* __restrict__ ids, int64_t n_tok,
                                                          const T* __restrict__ table, int64_t V, int64_t H,
                                                          int tp, T* __restrict__ out, int32_t* err) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int N = V16<T>::N;
  const int64_t tok = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (tok >= n_tok) return;
  const int64_t id = ids[tok];
  const int64_t per = V / tp;
  const T* row = nullptr;
  for (int r = 0; r < tp; ++r) {
    const int64_t start = per * r;
    const bool mask = (id >= start) && (id < start + per);   // step 1
    const int64_t local = mask ? (id - start) : 0;            // step 2
    if (mask) row = table + (start + local) * H;              // step 3 (W_r[local]); others contribute 0 (step 4)
  }
  if (row == nullptr && lane == 0 && err != nullptr) atomicAdd(err, 1);
  T* o = out + tok * H;
  constexpr int UNR = 4;
  for (int64_t c0 = int64_t(lane) * N; c0 < H; c0 += 32 * N * UNR) {
    float f[UNR][N];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t c = c0 + int64_t(u) * 32 * N;
      if (c < H && row != nullptr) load16(row + c, f[u]);
      else {
#pragma unroll
        for (int e = 0; e < N; ++e) f[u][e] = 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int64_t c = c0 + int64_t(u) * 32 * N;
      if (c < H) {
#pragma unroll
        for (int e = 0; e < N; ++e) f[u][e] = 0.0f + f[u][e];   // step 5: sum with the zero rows
        store16(o + c, f[u]);
      }
    }
  }
}

// ===========================================================================
// fused residual add + RMSNorm  ([SK] §2)
// one warp per row; NV 16-byte vectors per lane held in registers.
// ===========================================================================
template <typename T, int NV>
__global__ void __launch_bounds__(256) add_rmsnorm_kernel(const T* __restrict__ x, const T* res_in, T* res_out,
                                                          const T* __restrict__ gamma, float eps, int64_t rows,
                                                          int H, T* __restrict__ y) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int N = V16<T>::N;
  const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nvec = H / N;
  const int64_t base = row * H;
  float v[NV][N];
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vi = lane + 32 * i;
    if (vi < nvec) {
      load16(x + base + vi * N, v[i]);
      if (res_in != nullptr) {
        float r[N];
        load16(res_in + base + vi * N, r);
#pragma unroll
        for (int e = 0; e < N; ++e) v[i][e] = round_t<T>(v[i][e] + r[e]);   // x = x + residual (model dtype)
      }
      if (res_out != nullptr) store16(res_out + base + vi * N, v[i]);        // residual = x
#pragma unroll
      for (int e = 0; e < N; ++e) ss += v[i][e] * v[i][e];
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / float(H) + eps);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vi = lane + 32 * i;
    if (vi < nvec) {
      float g[N], o[N];
      load16(gamma + vi * N, g);
#pragma unroll
      for (int e = 0; e < N; ++e) o[e] = (v[i][e] * inv) * g[e];
      store16(y + base + vi * N, o);
    }
  }
}

// ===========================================================================
// QK-RMSNorm + RoPE + KV-cache store  ([SK] §8 ①, §3, §7.1)
// one warp per (token, head) over nh q heads then nkv kv heads; a kv-head
// warp also copies the raw v head into the cache.  RoPE pairs (i, i + hd/2)
// live in the same lane.
// ===========================================================================
template <typename T, int PPL>
__global__ void __launch_bounds__(256) qkv_norm_rope_kernel(
    const T* __restrict__ qkv, int64_t n_tok, int nh, int nkv, int hd, int tp,
    const int64_t* __restrict__ positions, const float* __restrict__ cos_sin, int64_t max_pos,
    const T* __restrict__ q_gamma, const T* __restrict__ k_gamma, float eps,
    const int64_t* __restrict__ slots, T* __restrict__ k_cache, T* __restrict__ v_cache, int64_t num_slots,
    T* __restrict__ q_out, int32_t* err) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int heads = nh + nkv;
  if (w >= n_tok * heads) return;
  const int64_t tok = w / heads;
  const int h = int(w % heads);
  const int nh_l = nh / tp, nkv_l = nkv / tp;
  const int64_t width_r = int64_t(nh_l + 2 * nkv_l) * hd;
  const int64_t row_w = width_r * tp;
  const bool is_q = h < nh;
  const T* src;
  const T* vsrc = nullptr;
  const T* gamma;
  int g = 0;
  if (is_q) {
    const int r = h / nh_l, hl = h % nh_l;
    src = qkv + tok * row_w + r * width_r + int64_t(hl) * hd;
    gamma = q_gamma;
  } else {
    g = h - nh;
    const int r = g / nkv_l, gl = g % nkv_l;
    src = qkv + tok * row_w + r * width_r + int64_t(nh_l + gl) * hd;
    vsrc = src + int64_t(nkv_l) * hd;
    gamma = k_gamma;
  }
  const int half = hd >> 1;
  float x1[PPL], x2[PPL];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < PPL; ++j) {
    const int i = lane + 32 * j;
    x1[j] = x2[j] = 0.0f;
    if (i < half) {
      x1[j] = to_f(src[i]);
      x2[j] = to_f(src[i + half]);
      ss += x1[j] * x1[j] + x2[j] * x2[j];
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / float(hd) + eps);
  const int64_t pos = positions[tok];
  const bool pos_ok = pos >= 0 && pos < max_pos;
  if (!pos_ok && lane == 0 && h == 0 && err != nullptr) atomicAdd(err, 1);
  const float* cs = cos_sin + (pos_ok ? pos : 0) * hd;
  float y1[PPL], y2[PPL];
#pragma unroll
  for (int j = 0; j < PPL; ++j) {
    const int i = lane + 32 * j;
    y1[j] = y2[j] = 0.0f;
    if (i < half) {
      const float n1 = round_t<T>((x1[j] * inv) * to_f(gamma[i]));          // q_norm / k_norm output
      const float n2 = round_t<T>((x2[j] * inv) * to_f(gamma[i + half]));
      const float c = cs[i], s = cs[half + i];
      y1[j] = n1 * c - n2 * s;                                               // RoPE on the halves
      y2[j] = n2 * c + n1 * s;
      if (!pos_ok) y1[j] = y2[j] = 0.0f;
    }
  }
  if (is_q) {
    T* o = q_out + (tok * nh + h) * int64_t(hd);
#pragma unroll
    for (int j = 0; j < PPL; ++j) {
      const int i = lane + 32 * j;
      if (i < half) {
        o[i] = from_f<T>(y1[j]);
        o[i + half] = from_f<T>(y2[j]);
      }
    }
    return;
  }
  const int64_t slot = slots[tok];
  if (slot == -1) return;                                                    // padding: not stored
  if (slot < 0 || slot >= num_slots || !pos_ok) {
    if (lane == 0 && g == 0 && err != nullptr && (slot < 0 || slot >= num_slots)) atomicAdd(err, 1);
    return;
  }
  T* kd = k_cache + (slot * nkv + g) * int64_t(hd);
  T* vd = v_cache + (slot * nkv + g) * int64_t(hd);
#pragma unroll
  for (int j = 0; j < PPL; ++j) {
    const int i = lane + 32 * j;
    if (i < half) {
      kd[i] = from_f<T>(y1[j]);
      kd[i + half] = from_f<T>(y2[j]);
    }
  }
  for (int e = lane; e < hd; e += 32) vd[e] = vsrc[e];                       // v: bit copy
}

// ===========================================================================
// QK-RMSNorm + RoPE + KV-cache store, bf16 with head_dim 128 (the model's
// shape): eight lanes per head.  Lane j of a group moves elements
// [8j, 8j+8) of the first half and [64+8j, 64+8j+8) of the second as 16-byte
// vectors, so every RoPE pair (i, i + 64) lives in one lane; the head's sum of
// squares is reduced over the eight lanes.  Same arithmetic as above.
// ===========================================================================
__global__ void __launch_bounds__(256) qkv_norm_rope_hd128_kernel(
    const bf16* __restrict__ qkv, int64_t n_tok, int nh, int nkv, int tp, const int64_t* __restrict__ positions,
    const float* __restrict__ cos_sin, int64_t max_pos, const bf16* __restrict__ q_gamma,
    const bf16* __restrict__ k_gamma, float eps, const int64_t* __restrict__ slots, bf16* __restrict__ k_cache,
    bf16* __restrict__ v_cache, int64_t num_slots, bf16* __restrict__ q_out, int32_t* err) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int HD = 128, HALF = 64;
  const int heads = nh + nkv;
  const int64_t task = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 3;   // one (token, head) per 8 lanes
  const int sub = threadIdx.x & 7;
  if (task >= n_tok * heads) return;   // whole 8-lane groups leave together
  const int64_t tok = task / heads;
  const int h = int(task % heads);
  const int nh_l = nh / tp, nkv_l = nkv / tp;
  const int64_t width_r = int64_t(nh_l + 2 * nkv_l) * HD;
  const int64_t row_w = width_r * tp;
  const bool is_q = h < nh;
  const bf16* src;
  const bf16* gamma;
  int g = 0;
  if (is_q) {
    src = qkv + tok * row_w + (h / nh_l) * width_r + int64_t(h % nh_l) * HD;
    gamma = q_gamma;
  } else {
    g = h - nh;
    src = qkv + tok * row_w + (g / nkv_l) * width_r + int64_t(nh_l + g % nkv_l) * HD;
    gamma = k_gamma;
  }
  const int i0 = 8 * sub;
  // every load that does not depend on another first: the position, the slot
  // and v (kv heads), the head's elements and gamma; then the RoPE row
  const int64_t pos = positions[tok];
  const int64_t slot = is_q ? -1 : slots[tok];
  uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
  if (!is_q) {
    const bf16* vs = src + int64_t(nkv_l) * HD;   // v: bit copy
    va = *reinterpret_cast<const uint4*>(vs + 2 * i0);
    vb = *reinterpret_cast<const uint4*>(vs + 2 * i0 + 8);
  }
  float x1[8], x2[8];
  load16(src + i0, x1);
  load16(src + HALF + i0, x2);
  float g1[8], g2[8];
  load16(gamma + i0, g1);
  load16(gamma + HALF + i0, g2);
  const bool pos_ok = pos >= 0 && pos < max_pos;
  const float* cs = cos_sin + (pos_ok ? pos : 0) * HD;
  float c[8], sn[8];
  *reinterpret_cast<float4*>(c) = *reinterpret_cast<const float4*>(cs + i0);
  *reinterpret_cast<float4*>(c + 4) = *reinterpret_cast<const float4*>(cs + i0 + 4);
  *reinterpret_cast<float4*>(sn) = *reinterpret_cast<const float4*>(cs + HALF + i0);
  *reinterpret_cast<float4*>(sn + 4) = *reinterpret_cast<const float4*>(cs + HALF + i0 + 4);
  // lane `sub` holds partial `sub`; the xor tree forms qk_ss_tree's balanced sum in every lane
  float ss = qk_ss8(x1, x2);
  ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 1));
  ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 2));
  ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, 4));
  const float inv = qk_inv_rms(ss, eps);
  if (!pos_ok && sub == 0 && h == 0 && err != nullptr) atomicAdd(err, 1);
  float y1[8], y2[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qk_rope_pair(x1[e], x2[e], inv, g1[e], g2[e], c[e], sn[e], pos_ok, y1[e], y2[e]);
  if (is_q) {
    bf16* o = q_out + (tok * nh + h) * int64_t(HD);
    store16(o + i0, y1);
    store16(o + HALF + i0, y2);
    return;
  }
  if (slot == -1) return;                                                    // padding: not stored
  if (slot < 0 || slot >= num_slots || !pos_ok) {
    if (sub == 0 && g == 0 && err != nullptr && (slot < 0 || slot >= num_slots)) atomicAdd(err, 1);
    return;
  }
  bf16* kd = k_cache + (slot * nkv + g) * int64_t(HD);
  bf16* vd = v_cache + (slot * nkv + g) * int64_t(HD);
  store16(kd + i0, y1);
  store16(kd + HALF + i0, y2);
  *reinterpret_cast<uint4*>(vd + 2 * i0) = va;
  *reinterpret_cast<uint4*>(vd + 2 * i0 + 8) = vb;
}

// ===========================================================================
// SiluAndMul  ([SK] §4): out[:, r*I_l + j] = silu(gate_r[j]) * up_r[j]
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(256) silu_mul_kernel(const T* __restrict__ x, T* __restrict__ out,
                                                       int64_t n_tok, int64_t I, int64_t I_l) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int N = V16<T>::N;
  const int64_t vpr = I / N;
  const int64_t idx = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= n_tok * vpr) return;
  const int64_t t = idx / vpr;
  const int64_t c = (idx % vpr) * N;
  const int64_t r = c / I_l, j = c % I_l;
  const T* gp = x + t * 2 * I + r * 2 * I_l + j;
  float gv[N], uv[N], o[N];
  load16(gp, gv);
  load16(gp + I_l, uv);
#pragma unroll
  for (int e = 0; e < N; ++e) o[e] = gv[e] / (1.0f + expf(-gv[e])) * uv[e];
  store16(out + t * I + c, o);
}

// ===========================================================================
// greedy argmax over a logits row, lowest index on ties
// ===========================================================================
// A row is split over a cluster of AM_CLUSTER CTAs (contiguous index ranges
// in rank order); each CTA reduces its range, and cluster rank 0 combines the
// CTAs' (max, index) pairs in rank order over distributed shared memory.  Every
// comparison keeps the lower index on equal values, so the result is the
// first maximum of the row.
constexpr int AM_CLUSTER = 8, AM_THREADS = 256, AM_UNROLL = 4;
template <typename T>
__global__ void __launch_bounds__(AM_THREADS) argmax_kernel(const T* __restrict__ logits, int64_t V,
                                                           int64_t* __restrict__ out) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int N = V16<T>::N;
  const int64_t row = blockIdx.x / AM_CLUSTER;
  const uint32_t rank = cluster_rank();
  const T* p = logits + row * V;
  const int64_t nv = V / N;   // (V * sizeof(T) is a multiple of 16 bytes)
  const int64_t per = (nv + AM_CLUSTER - 1) / AM_CLUSTER;
  const int64_t v0 = int64_t(rank) * per, v1 = min(nv, v0 + per);
  float best = -INFINITY;
  int64_t bidx = V;
  auto take = [&](float ob, int64_t oi) {
    if (ob > best || (ob == best && oi < bidx)) { best = ob; bidx = oi; }
  };
  for (int64_t vi = v0 + threadIdx.x; vi < v1; vi += AM_THREADS * AM_UNROLL) {
    float f[AM_UNROLL][N];
#pragma unroll
    for (int u = 0; u < AM_UNROLL; ++u)   // the loads of a pass in flight together
      if (vi + u * AM_THREADS < v1) load16(p + (vi + u * AM_THREADS) * N, f[u]);
#pragma unroll
    for (int u = 0; u < AM_UNROLL; ++u)
      if (vi + u * AM_THREADS < v1)
#pragma unroll
        for (int e = 0; e < N; ++e)
          if (f[u][e] > best) { best = f[u][e]; bidx = (vi + u * AM_THREADS) * N + e; }   // increasing index
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) take(__shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bidx, o));
  __shared__ float sb[AM_THREADS / 32];
  __shared__ int64_t si[AM_THREADS / 32];
  __shared__ float cb;      // this CTA's result, read by cluster rank 0
  __shared__ int64_t ci;
  const int wid = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sb[wid] = best; si[wid] = bidx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    best = sb[0];
    bidx = si[0];
    for (int w = 1; w < AM_THREADS / 32; ++w) take(sb[w], si[w]);
    cb = best;
    ci = bidx;
  }
  cluster_sync_all();   // every CTA's result is visible to the cluster
  if (rank == 0 && threadIdx.x == 0) {
    best = -INFINITY;
    bidx = V;
    for (uint32_t r = 0; r < AM_CLUSTER; ++r)
      take(ld_cluster_f32(map_to_rank(smem_u32(&cb), r)), ld_cluster_s64(map_to_rank(smem_u32(&ci), r)));
    out[row] = bidx < V ? bidx : 0;
  }
  cluster_sync_all();   // rank 0 has read every CTA's shared memory
}

// ===========================================================================
// row gather: out[i] = src[idx[i]]  (the prefill lm_head's last-token select)
// ===========================================================================
template <typename T>
__global__ void __launch_bounds__(256) gather_rows_kernel(const T* __restrict__ src, int64_t n_src,
                                                          const int32_t* __restrict__ idx, int64_t n,
                                                          int64_t H, T* __restrict__ out) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int N = V16<T>::N;
  const int64_t r = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= n) return;
  const int64_t s = idx[r];
  const bool ok = s >= 0 && s < n_src;
  for (int64_t c = int64_t(lane) * N; c < H; c += 32 * N) {
    float f[N];
    if (ok) load16(src + s * H + c, f);
    else {
#pragma unroll
      for (int e = 0; e < N; ++e) f[e] = 0.0f;
    }
    store16(out + r * H + c, f);
  }
}

template <typename T>
int launch_gather_rows(const void* src, int64_t n_src, const int32_t* idx, int64_t n, int64_t H, void* out,
                       cudaStream_t st) {
  const int64_t threads = n * 32;
  launch_pdl(gather_rows_kernel<T>, unsigned((threads + 255) / 256), 256, 0, st, 
      static_cast<const T*>(src), n_src, idx, n, H, static_cast<T*>(out));
  return check_launch("gather_rows");
}
template int launch_gather_rows<bf16>(const void*, int64_t, const int32_t*, int64_t, int64_t, void*, cudaStream_t);
template int launch_gather_rows<float>(const void*, int64_t, const int32_t*, int64_t, int64_t, void*, cudaStream_t);

template <typename T>
int launch_argmax(const void* logits, int64_t M, int64_t V, int64_t* out, cudaStream_t st) {
  if (M <= 0) return QW_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(M * AM_CLUSTER));
  cfg.blockDim = dim3(AM_THREADS);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = AM_CLUSTER;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, argmax_kernel<T>, static_cast<const T*>(logits), V, out);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "argmax launch: %s", cudaGetErrorString(e));
  return check_launch("argmax");
}
template int launch_argmax<bf16>(const void*, int64_t, int64_t, int64_t*, cudaStream_t);
template int launch_argmax<float>(const void*, int64_t, int64_t, int64_t*, cudaStream_t);

}  // namespace qw

// ===========================================================================
// C ABI
// ===========================================================================
using namespace qw;

static inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static inline size_t esize(int dtype) { return dtype == QW_BF16 ? 2 : 4; }

extern "C" int qw_embed_vocab(const int64_t* ids, int64_t T, const void* table, int64_t V, int64_t H, int tp,
                              void* out, int32_t* err_count, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_embed_vocab: dtype %d", dtype);
  if (T < 0 || V <= 0 || H <= 0 || tp <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_embed_vocab: bad sizes");
  if (V % tp != 0) return set_error(QW_ERR_SHAPE, "qw_embed_vocab: V=%lld not divisible by tp=%d", (long long)V, tp);
  if (T == 0) return QW_OK;
  if (!ids || !table || !out) return set_error(QW_ERR_INVALID_ARG, "qw_embed_vocab: null pointer");
  if ((H * esize(dtype)) % 16 || !al16(table) || !al16(out))
    return set_error(QW_ERR_INVALID_ARG, "qw_embed_vocab: rows must be 16-byte multiples and aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t threads = T * 32;
  const unsigned blocks = unsigned((threads + 255) / 256);
  if (dtype == QW_BF16)
    launch_pdl(embed_vocab_kernel<bf16>, blocks, 256, 0, st, ids, T, static_cast<const bf16*>(table), V, H, tp,
                                                     static_cast<bf16*>(out), err_count);
  else
    launch_pdl(embed_vocab_kernel<float>, blocks, 256, 0, st, ids, T, static_cast<const float*>(table), V, H, tp,
                                                      static_cast<float*>(out), err_count);
  return check_launch("qw_embed_vocab");
}

template <typename T>
static void launch_add_rmsnorm(int nv, const void* x, const void* ri, void* ro, const void* g, float eps,
                               int64_t T_, int H, void* y, cudaStream_t st) {
  const unsigned blocks = unsigned((T_ * 32 + 255) / 256);
  auto X = static_cast<const T*>(x);
  auto RI = static_cast<const T*>(ri);
  auto RO = static_cast<T*>(ro);
  auto G = static_cast<const T*>(g);
  auto Y = static_cast<T*>(y);
  switch (nv) {
    case 1: launch_pdl(add_rmsnorm_kernel<T, 1>, blocks, 256, 0, st, X, RI, RO, G, eps, T_, H, Y); break;
    case 2: launch_pdl(add_rmsnorm_kernel<T, 2>, blocks, 256, 0, st, X, RI, RO, G, eps, T_, H, Y); break;
    case 4: launch_pdl(add_rmsnorm_kernel<T, 4>, blocks, 256, 0, st, X, RI, RO, G, eps, T_, H, Y); break;
    case 8: launch_pdl(add_rmsnorm_kernel<T, 8>, blocks, 256, 0, st, X, RI, RO, G, eps, T_, H, Y); break;
    default: launch_pdl(add_rmsnorm_kernel<T, 16>, blocks, 256, 0, st, X, RI, RO, G, eps, T_, H, Y); break;
  }
}

extern "C" int qw_add_rmsnorm(const void* x, const void* residual_in, void* residual_out, const void* gamma,
                              float eps, int64_t T, int64_t H, void* y, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_add_rmsnorm: dtype %d", dtype);
  if (T < 0 || H <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm: bad sizes");
  if (T == 0) return QW_OK;
  if (!x || !gamma || !y) return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm: null pointer");
  const int N = int(16 / esize(dtype));
  if (H % N || !al16(x) || !al16(gamma) || !al16(y) || (residual_in && !al16(residual_in)) ||
      (residual_out && !al16(residual_out)))
    return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm: H must fill 16-byte vectors, pointers 16-byte aligned");
  const int64_t nvec = H / N;
  if (nvec > 32 * 16) return set_error(QW_ERR_SHAPE, "qw_add_rmsnorm: H=%lld too large", (long long)H);
  if (y == x || y == residual_in) return set_error(QW_ERR_INVALID_ARG, "qw_add_rmsnorm: y aliases an input");
  int nv = 1;
  while (nv * 32 < nvec) nv *= 2;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == QW_BF16) launch_add_rmsnorm<bf16>(nv, x, residual_in, residual_out, gamma, eps, T, int(H), y, st);
  else launch_add_rmsnorm<float>(nv, x, residual_in, residual_out, gamma, eps, T, int(H), y, st);
  return check_launch("qw_add_rmsnorm");
}

extern "C" int qw_rope_cos_sin_table(float* host_out, int64_t max_position, int rotary_dim, double theta) {
  if (!host_out || max_position <= 0 || rotary_dim <= 0 || (rotary_dim & 1) || !(theta > 0))
    return set_error(QW_ERR_INVALID_ARG, "qw_rope_cos_sin_table: bad arguments");
  const int half = rotary_dim / 2;
  for (int i = 0; i < half; ++i) {
    // inv_freq_i = 1 / theta^(2i/d), the exact value rounded to fp32
    const float inv_freq = float(1.0 / pow(theta, double(2 * i) / double(rotary_dim)));
    for (int64_t p = 0; p < max_position; ++p) {
      const float angle = float(p) * inv_freq;                  // fp32 product, as the fp32 outer product
      host_out[p * rotary_dim + i] = float(cos(double(angle)));
      host_out[p * rotary_dim + half + i] = float(sin(double(angle)));
    }
  }
  return QW_OK;
}

template <typename T>
static void launch_qkv_rope(int ppl, const void* qkv, int64_t T_, int nh, int nkv, int hd, int tp,
                            const int64_t* pos, const float* cs, int64_t maxp, const void* qg, const void* kg,
                            float eps, const int64_t* slots, void* kc, void* vc, int64_t ns, void* qo,
                            int32_t* err, cudaStream_t st) {
  const int64_t threads = T_ * (nh + nkv) * 32;
  const unsigned blocks = unsigned((threads + 255) / 256);
  auto a = static_cast<const T*>(qkv);
  auto g1 = static_cast<const T*>(qg);
  auto g2 = static_cast<const T*>(kg);
  auto k = static_cast<T*>(kc);
  auto v = static_cast<T*>(vc);
  auto q = static_cast<T*>(qo);
  switch (ppl) {
    case 1: launch_pdl(qkv_norm_rope_kernel<T, 1>, blocks, 256, 0, st, a, T_, nh, nkv, hd, tp, pos, cs, maxp, g1, g2, eps, slots, k, v, ns, q, err); break;
    case 2: launch_pdl(qkv_norm_rope_kernel<T, 2>, blocks, 256, 0, st, a, T_, nh, nkv, hd, tp, pos, cs, maxp, g1, g2, eps, slots, k, v, ns, q, err); break;
    case 3: launch_pdl(qkv_norm_rope_kernel<T, 3>, blocks, 256, 0, st, a, T_, nh, nkv, hd, tp, pos, cs, maxp, g1, g2, eps, slots, k, v, ns, q, err); break;
    default: launch_pdl(qkv_norm_rope_kernel<T, 4>, blocks, 256, 0, st, a, T_, nh, nkv, hd, tp, pos, cs, maxp, g1, g2, eps, slots, k, v, ns, q, err); break;
  }
}

extern "C" int qw_qkv_norm_rope_store_kv(const void* qkv, int64_t T, int n_heads, int n_kv_heads, int head_dim,
                                         int tp, const int64_t* positions, const float* cos_sin,
                                         int64_t max_position, const void* q_gamma, const void* k_gamma, float eps,
                                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                         int64_t num_slots, void* q_out, int32_t* err_count, int dtype,
                                         void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_qkv_norm_rope_store_kv: dtype %d", dtype);
  if (T < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || tp <= 0 || max_position <= 0 || num_slots < 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_qkv_norm_rope_store_kv: bad sizes");
  if (n_heads % tp || n_kv_heads % tp || (head_dim & 1) || head_dim > 256)
    return set_error(QW_ERR_SHAPE, "qw_qkv_norm_rope_store_kv: nh=%d nkv=%d hd=%d tp=%d", n_heads, n_kv_heads,
                     head_dim, tp);
  if (T == 0) return QW_OK;
  if (!qkv || !positions || !cos_sin || !q_gamma || !k_gamma || !slot_mapping || !k_cache || !v_cache || !q_out)
    return set_error(QW_ERR_INVALID_ARG, "qw_qkv_norm_rope_store_kv: null pointer");
  const int ppl = (head_dim / 2 + 31) / 32;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool aligned = (reinterpret_cast<uintptr_t>(qkv) | reinterpret_cast<uintptr_t>(q_out) |
                        reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
                        reinterpret_cast<uintptr_t>(cos_sin) | reinterpret_cast<uintptr_t>(q_gamma) |
                        reinterpret_cast<uintptr_t>(k_gamma)) % 16 == 0;
  if (dtype == QW_BF16 && head_dim == 128 && aligned) {
    const int64_t threads = T * (n_heads + n_kv_heads) * 8;
    launch_pdl(qkv_norm_rope_hd128_kernel, unsigned((threads + 255) / 256), 256, 0, st,
               static_cast<const bf16*>(qkv), T, n_heads, n_kv_heads, tp, positions, cos_sin, max_position,
               static_cast<const bf16*>(q_gamma), static_cast<const bf16*>(k_gamma), eps, slot_mapping,
               static_cast<bf16*>(k_cache), static_cast<bf16*>(v_cache), num_slots, static_cast<bf16*>(q_out),
               err_count);
    return check_launch("qw_qkv_norm_rope_store_kv");
  }
  if (dtype == QW_BF16)
    launch_qkv_rope<bf16>(ppl, qkv, T, n_heads, n_kv_heads, head_dim, tp, positions, cos_sin, max_position, q_gamma,
                          k_gamma, eps, slot_mapping, k_cache, v_cache, num_slots, q_out, err_count, st);
  else
    launch_qkv_rope<float>(ppl, qkv, T, n_heads, n_kv_heads, head_dim, tp, positions, cos_sin, max_position, q_gamma,
                           k_gamma, eps, slot_mapping, k_cache, v_cache, num_slots, q_out, err_count, st);
  return check_launch("qw_qkv_norm_rope_store_kv");
}

extern "C" int qw_silu_mul(const void* x, void* out, int64_t T, int64_t I, int tp, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_silu_mul: dtype %d", dtype);
  if (T < 0 || I <= 0 || tp <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_silu_mul: bad sizes");
  const int N = int(16 / esize(dtype));
  if (I % tp || (I / tp) % N) return set_error(QW_ERR_SHAPE, "qw_silu_mul: I=%lld tp=%d", (long long)I, tp);
  if (T == 0) return QW_OK;
  if (!x || !out || !al16(x) || !al16(out)) return set_error(QW_ERR_INVALID_ARG, "qw_silu_mul: null or misaligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n = T * (I / N);
  const unsigned blocks = unsigned((n + 255) / 256);
  if (dtype == QW_BF16)
    launch_pdl(silu_mul_kernel<bf16>, blocks, 256, 0, st, static_cast<const bf16*>(x), static_cast<bf16*>(out), T, I, I / tp);
  else
    launch_pdl(silu_mul_kernel<float>, blocks, 256, 0, st, static_cast<const float*>(x), static_cast<float*>(out), T, I,
                                                    I / tp);
  return check_launch("qw_silu_mul");
}

extern "C" int qw_argmax(const void* logits, int64_t M, int64_t V, int64_t* out, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_argmax: dtype %d", dtype);
  if (M < 0 || V <= 0) return set_error(QW_ERR_INVALID_ARG, "qw_argmax: bad sizes");
  if (M == 0) return QW_OK;
  if (!logits || !out || !al16(logits) || (V * esize(dtype)) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_argmax: null/misaligned logits or V not a 16-byte multiple");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return dtype == QW_BF16 ? launch_argmax<bf16>(logits, M, V, out, st) : launch_argmax<float>(logits, M, V, out, st);
}
