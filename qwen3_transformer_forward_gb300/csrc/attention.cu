// Causal GQA attention of the Qwen3 forward pass ([SK] §7.2): the CUDA-core
// path for small head_dim (prefill and decode) and decode over the KV cache.
// (Prefill with head_dim 128 runs on tcgen05 tensor cores: attention_prefill.cu.)
//
// Decode (head_dim 128): split-KV, each cached K/V byte read once, all q heads
// of a GQA group served together.
//   bf16: one persistent wave (attn_decode_tc_kernel).  CTAs take contiguous
//   ranges of the (sequence, kv head, 64-key tile) sequence, stream the tiles
//   through a TMA ring and run QK^T / PV on mma.sync.  Options: the QK-norm +
//   RoPE + KV store folded in (qw_attention_decode_rope), a paged cache
//   (qw_attention_decode_paged), history copies started before the
//   programmatic wait (QW_DECODE_HISTORY_READY).
//   f32: one CTA per (key chunk, kv head, sequence) over a cp.async double
//   buffer.
// In both, a (sequence, kv head) split over several CTAs leaves partial
// (m, l, o) in the caller's workspace.  The last to finish, by an atomic
// completion counter, merges them and writes the output.
// The paged prefill entry (qw_attention_prefill_paged) is also here; its kernel
// is in attention_prefill.cu.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace qw {
namespace attn {

constexpr float kLog2e = 1.4426950408889634f;

// Error word of the decode kernels: bits 0x1/0x2 record a bounded wait that gave up.
__device__ unsigned int g_attn_timeout = 0;
// Bit kErrContextOverflow (common.cuh) records a context length beyond max_context.

// ---------------------------------------------------------------------------
// tensor-core helpers (legacy warp-level MMA)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------------------
// small head_dim (<= 64), any dtype: one warp per (query token, q head).
// Prefill: query i of sequence s sees keys 0 .. Lk - Lq + i.  Decode
// (ctx_lens != nullptr): one query per sequence that sees ctx_lens[s] keys.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(128) attn_small_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_k, const int32_t* __restrict__ seq_base,
    const int32_t* __restrict__ ctx_lens, int n_seqs, int max_q, int nh, int nkv, int hd, float scale,
    T* __restrict__ out) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  const int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= int64_t(n_seqs) * max_q * nh) return;
  const int s = int(w / (int64_t(max_q) * nh));
  const int i = int((w / nh) % max_q);
  const int h = int(w % nh);
  int Lq, Lk;
  int64_t t;
  if (ctx_lens != nullptr) {
    Lq = 1;
    Lk = ctx_lens[s];
    t = s;
  } else {
    Lq = cu_q[s + 1] - cu_q[s];
    Lk = cu_k[s + 1] - cu_k[s];
    t = int64_t(cu_q[s]) + i;
  }
  if (i >= Lq) return;
  const int last = Lk - Lq + i;   // last visible key
  const int g = h / (nh / nkv);
  const int64_t kbase = seq_base != nullptr ? int64_t(seq_base[s]) : int64_t(cu_k[s]);
  const T* qv = q + (t * nh + h) * int64_t(hd);
  float m = -INFINITY, l = 0.0f;
  float acc0 = 0.0f, acc1 = 0.0f;   // lane owns d = lane and d = lane + 32
  for (int j0 = 0; j0 <= last; j0 += 32) {
    const int j = j0 + lane;
    float sc = -INFINITY;
    if (j <= last) {
      const T* kv = k + ((kbase + j) * nkv + g) * int64_t(hd);
      float d = 0.0f;
      for (int e = 0; e < hd; ++e) d = fmaf(to_f(qv[e]), to_f(kv[e]), d);
      sc = d * scale;
    }
    const float mt = warp_max(sc);
    const float m_new = fmaxf(m, mt);
    const float alpha = expf(m - m_new);
    const float p = j <= last ? expf(sc - m_new) : 0.0f;
    l = l * alpha + warp_sum(p);
    acc0 *= alpha;
    acc1 *= alpha;
    for (int jj = 0; jj < 32 && j0 + jj <= last; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const T* vv = v + ((kbase + j0 + jj) * nkv + g) * int64_t(hd);
      if (lane < hd) acc0 = fmaf(pj, to_f(vv[lane]), acc0);
      if (lane + 32 < hd) acc1 = fmaf(pj, to_f(vv[lane + 32]), acc1);
    }
    m = m_new;
  }
  T* o = out + (t * nh + h) * int64_t(hd);
  const float inv = l > 0.0f ? 1.0f / l : 0.0f;
  if (lane < hd) o[lane] = from_f<T>(acc0 * inv);
  if (lane + 32 < hd) o[lane + 32] = from_f<T>(acc1 * inv);
}

template <typename T>
int launch_attn_small(const void* q, const void* k, const void* v, const int32_t* cu_q, const int32_t* cu_k,
                      const int32_t* seq_base, const int32_t* ctx_lens, int n_seqs, int max_q, int nh, int nkv,
                      int hd, float scale, void* out, cudaStream_t st) {
  const int64_t threads = int64_t(n_seqs) * max_q * nh * 32;
  launch_pdl(attn_small_kernel<T>, unsigned((threads + 127) / 128), 128, 0, st, 
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), cu_q, cu_k, seq_base, ctx_lens,
      n_seqs, max_q, nh, nkv, hd, scale, static_cast<T*>(out));
  return check_launch("attn_small_kernel");
}

// ---------------------------------------------------------------------------
// decode: split-KV over the cache
// ---------------------------------------------------------------------------
constexpr int DC_HD = 128, DC_KT = 64, DC_THREADS = 128;

template <typename T>
constexpr size_t decode_smem() {
  return 2 * 2 * size_t(DC_KT) * DC_HD * sizeof(T);
}

// element e of row r in a swizzled [rows][128] tile of T
template <typename T>
__device__ __forceinline__ int dswz(int r, int e) {
  constexpr int EPC = 16 / sizeof(T);
  const int c = e / EPC;
  return r * DC_HD + ((c ^ (r & 7)) * EPC) + (e % EPC);
}

// Counts this chunk as done for its (sequence, kv head); the last chunk to
// finish merges every chunk's (m, l, o) for the group's q heads, writes the
// output and resets the counter.  All DC_THREADS threads call it.
template <typename T, int G>
__device__ __forceinline__ void decode_finish(const float* ws_o, const float* ws_ml, unsigned int* counters, int b,
                                              int g, int nh, int nkv, int n_splits, T* out) {
  constexpr int MAXS = 64;   // chunks per (sequence, kv head) merged through shared memory at a time
  __shared__ int s_last;
  __shared__ float s_w[G][MAXS];
  __shared__ float s_scale[G];
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    s_last = atomicAdd(counters + (int64_t(b) * nkv + g), 1u) == unsigned(n_splits - 1) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int d = threadIdx.x;
  const int64_t hrow0 = int64_t(b) * nh + int64_t(g) * G;
  float acc[G];
#pragma unroll
  for (int j = 0; j < G; ++j) acc[j] = 0.0f;
  float run_m[G], run_l[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    run_m[j] = -INFINITY;
    run_l[j] = 0.0f;
  }
  for (int s0 = 0; s0 < n_splits; s0 += MAXS) {
    const int ns = min(MAXS, n_splits - s0);
    // one warp per head: chunk maxima and weights relative to the running max
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < G; j += DC_THREADS / 32) {
      const int64_t hrow = hrow0 + j;
      float ms[2], ls[2];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int sp = lane + 32 * u;
        ms[u] = sp < ns ? __ldcg(ws_ml + 2 * (hrow * n_splits + s0 + sp)) : -INFINITY;
        ls[u] = sp < ns ? __ldcg(ws_ml + 2 * (hrow * n_splits + s0 + sp) + 1) : 0.0f;
        mx = fmaxf(mx, ms[u]);
      }
      mx = warp_max(mx);
      const float m_new = fmaxf(run_m[j], mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      float lsum = 0.0f;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float w = ms[u] == -INFINITY ? 0.0f : exp2f(ms[u] - m_use);
        if (lane + 32 * u < ns) s_w[j][lane + 32 * u] = w;
        lsum += ls[u] * w;
      }
      lsum = warp_sum(lsum);
      if (lane == 0) s_scale[j] = run_m[j] == -INFINITY ? 0.0f : exp2f(run_m[j] - m_use);
      run_l[j] = run_l[j] * (run_m[j] == -INFINITY ? 0.0f : exp2f(run_m[j] - m_use)) + lsum;
      run_m[j] = m_new;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int64_t hrow = hrow0 + j;
      float o = acc[j] * s_scale[j];
#pragma unroll 8
      for (int sp = 0; sp < ns; ++sp) o += __ldcg(ws_o + (hrow * n_splits + s0 + sp) * DC_HD + d) * s_w[j][sp];
      acc[j] = o;
    }
    __syncthreads();
  }
  // the warp that owned head j holds its running sum; publish it through shared memory
  __shared__ float s_l[G];
  {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < G; j += DC_THREADS / 32)
      if (lane == 0) s_l[j] = run_l[j];
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < G; ++j) out[(hrow0 + j) * DC_HD + d] = from_f<T>(s_l[j] > 0.0f ? acc[j] / s_l[j] : 0.0f);
  __syncthreads();
  if (threadIdx.x == 0) counters[int64_t(b) * nkv + g] = 0u;
}

template <typename T, int G>
__global__ void __launch_bounds__(DC_THREADS) attn_decode_kernel(
    const T* __restrict__ q, const T* __restrict__ kc, const T* __restrict__ vc, const int32_t* __restrict__ ctx_lens,
    const int32_t* __restrict__ seq_base, int nh, int nkv, float scale_log2, int chunk, int n_splits,
    float* __restrict__ ws_o, float* __restrict__ ws_ml, unsigned int* __restrict__ counters, T* __restrict__ out) {
  pdl_wait();      // inputs of this kernel are complete and visible
  pdl_trigger();   // only now may the next kernel start its prologue
  constexpr int EPC = 16 / sizeof(T);      // elements per 16-byte chunk
  constexpr int CPR = DC_HD / EPC;         // chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  T* sK = reinterpret_cast<T*>(smem);
  T* sV = sK + 2 * DC_KT * DC_HD;
  __shared__ float sQ[G][DC_HD];
  __shared__ float sS[G][DC_KT];
  __shared__ float sAlpha[G];
  __shared__ float sM[G], sL[G];
  __shared__ float sO[G][DC_HD];

  const int b = blockIdx.z, g = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int L = ctx_lens[b];
  if (tid == 0 && split == n_splits - 1 && L > n_splits * chunk) atomicOr(&g_attn_timeout, kErrContextOverflow);
  const int start = split * chunk;
  const int end = min(L, start + chunk);
  const int h0 = g * G;
  const int64_t row_stride = int64_t(nkv) * DC_HD;
  const int64_t base = seq_base[b];

  if (start >= end) {
    if (n_splits > 1) {
      if (tid < G) {
        const int64_t idx = (int64_t(b) * nh + h0 + tid) * n_splits + split;
        ws_ml[2 * idx] = -INFINITY;
        ws_ml[2 * idx + 1] = 0.0f;
      }
      decode_finish<T, G>(ws_o, ws_ml, counters, b, g, nh, nkv, n_splits, out);
    } else {
      for (int i = tid; i < G * DC_HD; i += DC_THREADS)
        out[(int64_t(b) * nh + h0 + i / DC_HD) * DC_HD + i % DC_HD] = from_f<T>(0.0f);
    }
    return;
  }
  for (int i = tid; i < G * DC_HD; i += DC_THREADS)
    sQ[i / DC_HD][i % DC_HD] = to_f(q[(int64_t(b) * nh + h0 + i / DC_HD) * DC_HD + i % DC_HD]);
  if (tid < G) {
    sM[tid] = -INFINITY;
    sL[tid] = 0.0f;
  }
  const int n_kt = (end - start + DC_KT - 1) / DC_KT;
  auto load = [&](int kt, int buf) {
    for (int i = tid; i < DC_KT * CPR; i += DC_THREADS) {
      const int r = i / CPR, c = i % CPR;
      const int key = start + kt * DC_KT + r;
      const bool ok = key < end;
      const int64_t off = (base + (ok ? key : start)) * row_stride + int64_t(g) * DC_HD + c * EPC;
      const int so = buf * DC_KT * DC_HD + r * DC_HD + ((c ^ (r & 7)) * EPC);
      cp_async16_zfill(smem_u32(sK + so), kc + off, ok);
      cp_async16_zfill(smem_u32(sV + so), vc + off, ok);
    }
  };
  load(0, 0);
  cp_async_commit();

  // PV ownership: dims d0, d0+1 for the keys of one half of the tile
  const int dpair = tid & 63, khalf = tid >> 6;
  float acc[G][2];
#pragma unroll
  for (int j = 0; j < G; ++j) acc[j][0] = acc[j][1] = 0.0f;

  for (int kt = 0; kt < n_kt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < n_kt) load(kt + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const T* tK = sK + buf * DC_KT * DC_HD;
    const T* tV = sV + buf * DC_KT * DC_HD;
    // scores: thread -> key (tid % 64), heads tid/64, tid/64 + 2, ...
    {
      const int kk = tid % DC_KT;
      const int key = start + kt * DC_KT + kk;
      for (int j = tid / DC_KT; j < G; j += DC_THREADS / DC_KT) {
        float d = 0.0f;
#pragma unroll 4
        for (int c = 0; c < CPR; ++c) {
          float f[EPC];
          load16(tK + kk * DC_HD + ((c ^ (kk & 7)) * EPC), f);
#pragma unroll
          for (int e = 0; e < EPC; ++e) d = fmaf(sQ[j][c * EPC + e], f[e], d);
        }
        sS[j][kk] = key < end ? d * scale_log2 : -INFINITY;
      }
    }
    __syncthreads();
    // online softmax: warp w handles heads w, w + 4
    for (int j = warp; j < G; j += DC_THREADS / 32) {
      const float s0 = sS[j][lane], s1 = sS[j][lane + 32];
      const float mt = warp_max(fmaxf(s0, s1));
      const float m_old = sM[j];
      const float m_new = fmaxf(m_old, mt);
      const float alpha = exp2f(m_old - m_new);       // m_new is finite: the tile has a valid key
      const float p0 = exp2f(s0 - m_new), p1 = exp2f(s1 - m_new);
      const float ps = warp_sum(p0 + p1);
      sS[j][lane] = p0;
      sS[j][lane + 32] = p1;
      if (lane == 0) {
        sM[j] = m_new;
        sL[j] = sL[j] * alpha + ps;
        sAlpha[j] = alpha;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float al = sAlpha[j];
      acc[j][0] *= al;
      acc[j][1] *= al;
    }
    const int d0 = 2 * dpair;
#pragma unroll 4
    for (int kk = khalf * 32; kk < khalf * 32 + 32; ++kk) {
      const float v0 = to_f(tV[dswz<T>(kk, d0)]);
      const float v1 = to_f(tV[dswz<T>(kk, d0 + 1)]);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float p = sS[j][kk];
        acc[j][0] = fmaf(p, v0, acc[j][0]);
        acc[j][1] = fmaf(p, v1, acc[j][1]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // combine the two key halves
  if (khalf == 1) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      sO[j][2 * dpair] = acc[j][0];
      sO[j][2 * dpair + 1] = acc[j][1];
    }
  }
  __syncthreads();
  if (khalf == 0) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float o0 = acc[j][0] + sO[j][2 * dpair];
      const float o1 = acc[j][1] + sO[j][2 * dpair + 1];
      const int64_t hrow = int64_t(b) * nh + h0 + j;
      if (n_splits > 1) {
        const int64_t idx = hrow * n_splits + split;
        ws_o[idx * DC_HD + 2 * dpair] = o0;
        ws_o[idx * DC_HD + 2 * dpair + 1] = o1;
        if (dpair == 0) {
          ws_ml[2 * idx] = sM[j];
          ws_ml[2 * idx + 1] = sL[j];
        }
      } else {
        const float inv = 1.0f / sL[j];
        out[hrow * DC_HD + 2 * dpair] = from_f<T>(o0 * inv);
        out[hrow * DC_HD + 2 * dpair + 1] = from_f<T>(o1 * inv);
      }
    }
  }
  if (n_splits > 1) decode_finish<T, G>(ws_o, ws_ml, counters, b, g, nh, nkv, n_splits, out);
}

// ---------------------------------------------------------------------------
// decode, bf16: tensor-core split-KV in one persistent wave.
//
// The work is laid out as a fixed grid of 64-key tiles: pair p = b * nkv + g
// (sequence b, kv head g) owns tiles [p * T, (p + 1) * T), T = ceil(max
// context / 64).  CTA c takes the contiguous range [c * per, (c + 1) * per)
// of that grid (per = ceil(P * T / gridDim)), so the split depends only on
// sizes the host knows and a CTA can start its copies at once; tiles at or
// past a sequence's own length are skipped.  K/V tiles arrive by TMA (3-D map
// over the cache [slot][kv head][dim], two 64-dim boxes with 128-byte swizzle
// each) through a 3-stage mbarrier ring that runs on across pair boundaries.
// Warp w owns keys 16w..16w+15 of every tile and runs its own online softmax:
// S = Q K^T and O += P V with mma.sync m16n8k16 (the group's G q heads padded
// to 16 rows).  At the end of each pair segment the four warps merge in
// shared memory.  A pair inside one CTA's range is written out directly;
// otherwise each of its CTAs c_first..c_last leaves (m, l, o) in workspace
// slot c + p (distinct for every (CTA, pair) that occurs, since a later CTA
// starts at or after the pair where an earlier one stopped), and the last to
// finish, by the pair's completion counter, merges them in CTA order.
// ---------------------------------------------------------------------------

constexpr int DT_KT = 64, DT_STAGES = 3, DT_THREADS = 128;
// History tiles copied ahead of the programmatic wait (<= DT_STAGES).  Two
// rather than a full ring leave more of the memory system to the previous
// kernel's tail: back to back 15.1 -> 14.7 us per launch, the decode step unchanged.
constexpr int DT_PRE = 2;
constexpr uint32_t DT_BOX = 64 * 64 * 2;          // 64 keys x 64 dims of bf16
constexpr uint32_t DT_STAGE = 4 * DT_BOX;         // K dims 0-63, K 64-127, V 0-63, V 64-127
constexpr int DT_MERGE = 8;                       // segments whose partials one merge step loads at once

// dynamic shared memory (after rounding the base up to 1024 B):
// ring | sO [4 warps][G][128] f32 | sML [4][G][2] f32 | flag | barriers
template <int G>
constexpr size_t dt_smem() {
  return 1024 + size_t(DT_STAGES) * DT_STAGE + size_t(4) * G * DC_HD * 4 + size_t(4) * G * 2 * 4 + 16 +
         2 * DT_STAGES * 8;
}

// byte offset of (key row r, 16-byte chunk c16 over the 128 dims) in a K or V region
__device__ __forceinline__ uint32_t kv_off(int r, int c16) {
  return uint32_t(c16 >> 3) * DT_BOX + uint32_t(r) * 128u + uint32_t(((c16 & 7) ^ (r & 7)) * 16);
}

__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int* p, unsigned int v) {
  unsigned int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The QK-RMSNorm + RoPE + KV store of the decode step ([SK] §3, §7.1, §8),
// folded into the decode kernel: the q heads come from the merged QKV output,
// and the CTA holding a pair's last tile stores that kv head's new k (normed,
// roped) and v before it loads the tile.  qkv == nullptr: q is read as given.
struct DecodeRope {
  const bf16* qkv;            // [B, tp * (nh/tp + 2 nkv/tp) * 128], shard r = [q_r; k_r; v_r]
  const int64_t* positions;   // [B]
  const int64_t* slots;       // [B]: cache row of this step's k/v; -1 = not stored
  const float* cos_sin;       // [max_pos, 128]: cos | sin
  int64_t max_pos;
  const bf16* q_gamma;        // [128]
  const bf16* k_gamma;        // [128]
  float eps;
  int tp;
  int32_t* err;               // counts bad positions and slots (may be null)
  bf16* k_cache;
  bf16* v_cache;
  int64_t num_slots;
};

template <int G>
__global__ void __launch_bounds__(DT_THREADS) attn_decode_tc_kernel(
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, const bf16* __restrict__ q,
    const int32_t* __restrict__ ctx_lens, const int32_t* __restrict__ seq_base, int nh, int nkv, int n_pairs,
    int T, int per, float scale_log2, int history_ready, float* __restrict__ ws_o, float* __restrict__ ws_ml,
    unsigned int* __restrict__ counters, bf16* __restrict__ out, const DecodeRope rp, const KvPages pages) {
  // history_ready: context lengths, bases and every cached row but each
  // sequence's last were complete before the previous kernel started, which
  // writes only q and those last rows.  Then the lengths are read and the
  // copies of tiles before each sequence's last start ahead of the wait.
  if (!history_ready) {
    pdl_wait();      // inputs of this kernel are complete and visible
    pdl_trigger();   // only now may the next kernel start its prologue
  }
  const int64_t lo = int64_t(blockIdx.x) * per;
  const int64_t hi = min(int64_t(n_pairs) * T, lo + per);
  if (lo >= hi) {   // uniform over the CTA
    if (history_ready) {
      pdl_wait();
      pdl_trigger();
    }
    return;
  }
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  float* sO = reinterpret_cast<float*>(sm + DT_STAGES * DT_STAGE);   // [4][G][128]
  float* sML = sO + 4 * G * DC_HD;                                   // [4][G][2]
  int* s_last = reinterpret_cast<int*>(sML + 4 * G * 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(s_last + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p_first = int(lo / T), p_last = int((hi - 1) / T);
  const int L_first = ctx_lens[p_first / nkv];   // loaded together with the base below
  const int base_first = pages.table == nullptr ? seq_base[p_first / nkv] : 0;
  // the folded QK-norm + RoPE's constants, in the same round trip: the first
  // sequence's position and both gammas (ahead of the wait with history_ready,
  // which covers positions; the weights are constants)
  const int d = tid;
  int64_t pos_first = 0;
  float gam_q = 0.0f, gam_k = 0.0f;
  if (rp.qkv != nullptr) {
    pos_first = rp.positions[p_first / nkv];
    gam_q = __bfloat162float(rp.q_gamma[d]);
    gam_k = __bfloat162float(rp.k_gamma[d]);
  }
  // this CTA's tiles of pair p: the static range clipped to the sequence's own length (Tb tiles)
  auto seg_range = [&](int p, int& ta, int& tb, int& Tb) {
    const int ts = p == p_first ? int(lo - int64_t(p) * T) : 0;
    const int te = p == p_last ? int(hi - int64_t(p) * T) : T;
    const int L = p / nkv == p_first / nkv ? L_first : ctx_lens[p / nkv];
    Tb = L > 0 ? (L + DT_KT - 1) / DT_KT : 0;
    ta = ts;
    tb = max(ts, min(te, Tb));
  };
  auto full = [&](int s) { return smem_u32(bars + s); };
  auto empty = [&](int s) { return smem_u32(bars + DT_STAGES + s); };

  // ---- producer state (thread 0): the next tile to load
  int pp = p_first, pt = 0, pt_end = 0, pTb = 0;
  auto prod_next = [&]() -> bool {   // moves to a pair with a tile left; false when none
    while (pt >= pt_end) {
      if (pp > p_last) return false;
      seg_range(pp, pt, pt_end, pTb);
      if (pt >= pt_end) ++pp;
    }
    return true;
  };
  int n_tiles = 0;   // tiles this CTA streams
  for (int p = p_first; p <= p_last; ++p) {
    int ta, tb, Tb;
    seg_range(p, ta, tb, Tb);
    n_tiles += tb - ta;
  }
  auto issue = [&](int j) {
    const int s = j % DT_STAGES;
    const uint32_t dst = smem_u32(sm + s * DT_STAGE);
    const int b = pp / nkv, g = pp % nkv;
    const int z = pages.table != nullptr   // cache row of key pt * 64, through the block table when paged
                      ? pages.table[int64_t(b) * pages.max_blocks + pt * DT_KT / pages.block_size] * pages.block_size +
                            (pt * DT_KT) % pages.block_size
                      : (b == p_first / nkv ? base_first : seq_base[b]) + pt * DT_KT;
    tcx::mbar_expect_tx(full(s), DT_STAGE);
    tcx::tma_load_3d(dst, &tmK, full(s), 0, g, z);
    tcx::tma_load_3d(dst + DT_BOX, &tmK, full(s), 64, g, z);
    tcx::tma_load_3d(dst + 2 * DT_BOX, &tmV, full(s), 0, g, z);
    tcx::tma_load_3d(dst + 3 * DT_BOX, &tmV, full(s), 64, g, z);
    if (++pt >= pt_end) ++pp;
  };
  int issued = 0;
  if (tid == 0) {
    for (int s = 0; s < DT_STAGES; ++s) {
      tcx::mbar_init(full(s), 1);
      tcx::mbar_init(empty(s), DT_THREADS / 32);
    }
    tcx::fence_mbar_init();
    // ahead of the wait: tiles before each sequence's last (which may still be written)
    if (history_ready)
      for (; issued < DT_PRE && issued < n_tiles; ++issued)
        if (!prod_next() || pt == pTb - 1) break;
        else issue(issued);
  }
  // ... and the first sequence's cos / sin, after the copies are on their
  // way, so that after the wait only the QKV row is a round trip
  float rope_c = 0.0f, rope_s = 0.0f;
  const bool pos_ok_first = pos_first >= 0 && pos_first < rp.max_pos;
  if (rp.qkv != nullptr) {
    const float* cs = rp.cos_sin + (pos_ok_first ? pos_first : 0) * DC_HD;
    rope_c = cs[d & 63];
    rope_s = cs[64 + (d & 63)];
  }
  if (history_ready) {
    pdl_wait();      // q and the sequences' last rows are complete and visible
    pdl_trigger();   // only now may the next kernel start its prologue
  }
  // ---- folded QK-norm + RoPE: head (sequence b, head slot h_off in a shard row) of
  // the QKV output normed by gamma, roped at positions[b] and rounded to bf16.
  // Thread d owns element d; RoPE pairs (d, d ^ 64) meet through shared memory.
  float* nrm = sO;                                           // [G][128] normed values
  bf16* qs = reinterpret_cast<bf16*>(sO + G * DC_HD);        // [G][128] roped q
  float* red = sML;                                          // [G][4] sums of squares
  const int nh_l = nh / rp.tp, nkv_l = nkv / rp.tp;
  const int64_t width_r = int64_t(nh_l + 2 * nkv_l) * DC_HD;
  auto norm_rope = [&](int b, const int64_t* h_off, float gm, int nheads, float* y) {
    const bf16* row = rp.qkv + int64_t(b) * width_r * rp.tp;
    float x[G];
#pragma unroll
    for (int j = 0; j < G; ++j)   // every head's element in flight at once
      if (j < nheads) x[j] = __bfloat162float(row[h_off[j] + d]);
    bool pos_ok = pos_ok_first;
    float c = rope_c, sn = rope_s;
    if (b != p_first / nkv) {   // a later sequence of this CTA's range
      const int64_t pos = rp.positions[b];
      pos_ok = pos >= 0 && pos < rp.max_pos;
      const float* cs = rp.cos_sin + (pos_ok ? pos : 0) * DC_HD;
      c = cs[d & 63];
      sn = cs[64 + (d & 63)];
    }
#pragma unroll
    for (int j = 0; j < G; ++j)
      if (j < nheads) {
        const float ss = warp_sum(x[j] * x[j]);
        if (lane == 0) red[j * 4 + warp] = ss;
      }
    __syncthreads();
    for (int j = 0; j < nheads; ++j) {
      const float ss = red[j * 4] + red[j * 4 + 1] + red[j * 4 + 2] + red[j * 4 + 3];
      const float inv = rsqrtf(ss / float(DC_HD) + rp.eps);
      nrm[j * DC_HD + d] = round_t<bf16>((x[j] * inv) * gm);   // q_norm / k_norm output
    }
    __syncthreads();
    for (int j = 0; j < nheads; ++j) {
      const float n = nrm[j * DC_HD + d], np = nrm[j * DC_HD + (d ^ 64)];
      y[j] = pos_ok ? (d < 64 ? n * c - np * sn : n * c + np * sn) : 0.0f;
    }
    __syncthreads();   // nrm and red are free again
    return pos_ok;
  };
  if (rp.qkv != nullptr) {
    // this CTA holds the last tile of pair p: store that kv head's new k and v
    for (int p = p_first; p <= p_last; ++p) {
      int ta, tb, Tb;
      seg_range(p, ta, tb, Tb);
      if (Tb == 0 || tb != Tb) continue;   // (uniform over the CTA)
      const int b = p / nkv, g = p % nkv;
      const int64_t k_off = int64_t(g / nkv_l) * width_r + int64_t(nh_l + g % nkv_l) * DC_HD;
      float y[G];
      const bool pos_ok = norm_rope(b, &k_off, gam_k, 1, y);
      const int64_t slot = rp.slots[b];
      if (slot != -1) {
        const bool slot_ok = slot >= 0 && slot < rp.num_slots;
        if (slot_ok && pos_ok) {
          rp.k_cache[(slot * nkv + g) * DC_HD + d] = __float2bfloat16_rn(y[0]);
          rp.v_cache[(slot * nkv + g) * DC_HD + d] = rp.qkv[int64_t(b) * width_r * rp.tp + k_off + int64_t(nkv_l) * DC_HD + d];
        }
        if (g == 0 && d == 0 && rp.err != nullptr && (!slot_ok || !pos_ok)) atomicAdd(rp.err, 1);
      }
    }
    // the stores above before the tensor copies that read them back
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __syncthreads();
  }
  if (tid == 0)
    for (int j = issued; j < DT_STAGES && j < n_tiles; ++j)
      if (prod_next()) issue(j);
  __syncthreads();

  const int gq = lane >> 2, tq = lane & 3;   // mma fragment row / column pair
  const int mi = lane >> 3, ri = lane & 7;   // ldmatrix matrix / row
  const int key0 = warp * 16;
  bool ok = true;
  int j = 0;   // ring position
  for (int p = p_first; p <= p_last; ++p) {
    const int b = p / nkv, g = p % nkv;
    int ta, tb, Tb;
    seg_range(p, ta, tb, Tb);
    if (tid == 0 && Tb > T) atomicOr(&g_attn_timeout, kErrContextOverflow);   // keys past max_context
    const int L = b == p_first / nkv ? L_first : ctx_lens[b];
    // q of this thread's row (head g * G + gq; rows >= G are zero)
    uint32_t qa[8][2];
    {
      const bf16* qr;
      if (rp.qkv == nullptr) {
        qr = q + (int64_t(b) * nh + g * G + (gq < G ? gq : 0)) * DC_HD;
      } else {   // QK-norm + RoPE of the group's q heads, into shared memory
        int64_t q_off[G];
#pragma unroll
        for (int jh = 0; jh < G; ++jh) {
          const int h = g * G + jh;
          q_off[jh] = int64_t(h / nh_l) * width_r + int64_t(h % nh_l) * DC_HD;
        }
        float y[G];
        norm_rope(b, q_off, gam_q, G, y);
#pragma unroll
        for (int jh = 0; jh < G; ++jh) qs[jh * DC_HD + d] = __float2bfloat16_rn(y[jh]);
        __syncthreads();
        qr = qs + (gq < G ? gq : 0) * DC_HD;
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        qa[kk][0] = gq < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * tq) : 0u;
        qa[kk][1] = gq < G ? *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 8 + 2 * tq) : 0u;
      }
    }
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    for (int t = ta; t < tb; ++t, ++j) {
      const int s = j % DT_STAGES;
      const uint32_t ph = (j / DT_STAGES) & 1;
      if (ok && !tcx::mbar_wait(full(s), ph, &g_attn_timeout, 1u)) ok = false;
      const uint32_t st = smem_u32(sm + s * DT_STAGE);
      const int kbase = t * DT_KT + key0;   // key position of this warp's first row
      if (kbase + 16 > L) {
        // keys past the sequence: zero their V rows (whatever the cache holds there)
        for (int i = 0; i < 16; ++i)
          if (kbase + i >= L && lane < 16)
            *reinterpret_cast<uint4*>(sm + s * DT_STAGE + 2 * DT_BOX + kv_off(key0 + i, lane)) =
                make_uint4(0, 0, 0, 0);
        tcx::fence_proxy_async();
        __syncwarp();
      }
      float sc[2][4];
#pragma unroll
      for (int nn = 0; nn < 2; ++nn) sc[nn][0] = sc[nn][1] = sc[nn][2] = sc[nn][3] = 0.0f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(st + kv_off(key0 + ri + 8 * (mi >> 1), 2 * kk + (mi & 1)), b0, b1, b2, b3);
        mma_bf16(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
        mma_bf16(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
      }
      float x[4];
      float mx = -INFINITY;
#pragma unroll
      for (int nn = 0; nn < 2; ++nn)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kp = kbase + 8 * nn + 2 * tq + e;
          const float v = kp < L ? sc[nn][e] * scale_log2 : -INFINITY;
          x[2 * nn + e] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = m_new == -INFINITY ? 0.0f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float pr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pr[i] = exp2f(x[i] - m_use);
      l_run = l_run * alpha + (pr[0] + pr[1] + pr[2] + pr[3]);
      m_run = m_new;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        o[i][0] *= alpha;
        o[i][1] *= alpha;
        o[i][2] *= alpha;
        o[i][3] *= alpha;
      }
      // P as two bf16 parts in the two row halves of the A fragment: rows 0-7
      // (the group's heads) hold hi = bf16(p), rows 8-15 (unused by the
      // heads) hold lo = bf16(p - hi), so accumulator rows 8-15 collect lo*V
      // at no extra MMA and hi + lo carries p to about 2^-17 relative.
      uint32_t a0, a1, a2, a3;
      split_p(pr, a0, a1, a2, a3);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(st + 2 * DT_BOX + kv_off(key0 + ri + 8 * (mi & 1), 2 * dp + (mi >> 1)), b0, b1, b2, b3);
        mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
      __syncwarp();
      if (lane == 0) tcx::mbar_arrive(empty(s));
      if (tid == 0 && j + DT_STAGES < n_tiles) {
        if (ok && !tcx::mbar_wait(empty(s), ph, &g_attn_timeout, 2u)) ok = false;
        // The warps read this stage with ldmatrix (generic proxy) and the copy
        // below overwrites it through the async proxy: the barrier alone does
        // not order the two proxies.  Without this fence a copy was seen to land
        // while a warp's last ldmatrix (V dims 112-127) was still pending.
        tcx::fence_proxy_async();
        if (ok && prod_next()) issue(j + DT_STAGES);
      }
    }
    // ---- end of this CTA's segment of pair p: merge the four warps' softmax states
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (gq < G) {
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {   // the hi and lo parts of P * V
        sO[(warp * G + gq) * DC_HD + 8 * dn + 2 * tq] = o[dn][0] + o[dn][2];
        sO[(warp * G + gq) * DC_HD + 8 * dn + 2 * tq + 1] = o[dn][1] + o[dn][3];
      }
      if (tq == 0) {
        sML[(warp * G + gq) * 2] = m_run;
        sML[(warp * G + gq) * 2 + 1] = l_run;
      }
    }
    __syncthreads();
    const int c_first = int(int64_t(p) * T / per), c_last = int((int64_t(p) * T + T - 1) / per);
    const bool split = c_first != c_last;
#pragma unroll
    for (int jh = 0; jh < G; ++jh) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < DT_THREADS / 32; ++w) M = fmaxf(M, sML[(w * G + jh) * 2]);
      float Lsum = 0.0f, O = 0.0f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < DT_THREADS / 32; ++w) {
          const float mw = sML[(w * G + jh) * 2];
          if (mw == -INFINITY) continue;
          const float scw = exp2f(mw - M);
          Lsum += sML[(w * G + jh) * 2 + 1] * scw;
          O += sO[(w * G + jh) * DC_HD + d] * scw;
        }
      }
      if (!split) {
        out[(int64_t(b) * nh + g * G + jh) * DC_HD + d] = __float2bfloat16_rn(Lsum > 0.0f ? O / Lsum : 0.0f);
      } else {
        const int64_t idx = (int64_t(blockIdx.x) + p) * G + jh;
        ws_o[idx * DC_HD + d] = O;
        if (d == 0) {
          ws_ml[2 * idx] = M;
          ws_ml[2 * idx + 1] = Lsum;
        }
      }
    }
    if (split) {
      // the CTA barrier orders every thread's partial before thread 0's
      // release; its acquire and the next barrier order the merge's reads
      __syncthreads();
      if (tid == 0) *s_last = atom_add_acq_rel_gpu(counters + p, 1u) == unsigned(c_last - c_first) ? 1 : 0;
      __syncthreads();
      if (*s_last) {
#pragma unroll
        for (int jh = 0; jh < G; ++jh) {
          float M = -INFINITY, Lsum = 0.0f, O = 0.0f;
          for (int c0 = c_first; c0 <= c_last; c0 += DT_MERGE) {
            float mc[DT_MERGE], lc[DT_MERGE], oc[DT_MERGE];
#pragma unroll
            for (int u = 0; u < DT_MERGE; ++u) {   // one batch of loads in flight together
              const int64_t idx = (int64_t(c0 + u) + p) * G + jh;
              const bool in = c0 + u <= c_last;
              mc[u] = in ? __ldcg(ws_ml + 2 * idx) : -INFINITY;
              lc[u] = in ? __ldcg(ws_ml + 2 * idx + 1) : 0.0f;
              oc[u] = in ? __ldcg(ws_o + idx * DC_HD + d) : 0.0f;
            }
            float mb = M;
#pragma unroll
            for (int u = 0; u < DT_MERGE; ++u) mb = fmaxf(mb, mc[u]);
            if (mb == -INFINITY) continue;
            const float rs = M == -INFINITY ? 0.0f : exp2f(M - mb);
            Lsum *= rs;
            O *= rs;
#pragma unroll
            for (int u = 0; u < DT_MERGE; ++u) {
              if (mc[u] == -INFINITY) continue;
              const float w = exp2f(mc[u] - mb);
              Lsum += lc[u] * w;
              O += oc[u] * w;
            }
            M = mb;
          }
          out[(int64_t(b) * nh + g * G + jh) * DC_HD + d] = __float2bfloat16_rn(Lsum > 0.0f ? O / Lsum : 0.0f);
        }
        if (tid == 0) counters[p] = 0u;
      }
    }
    __syncthreads();   // sO, sML and the flag are free for the next segment
  }
}

struct DecodePlan {
  int splits;
  int chunk;
};

inline DecodePlan decode_plan(int B, int max_context, int nkv_unused) {
  (void)nkv_unused;
  DecodePlan p{1, max_context > 0 ? max_context : 1};
  if (max_context <= 0) return p;
  // aim for >= ~4 CTAs per SM in total (152 SMs), keys chunks >= 128
  const int pairs = B * 8 > 0 ? B * 8 : 1;
  int s = (4 * 152 + pairs - 1) / pairs;
  const int smax = (max_context + 127) / 128;
  s = s < 1 ? 1 : (s > smax ? smax : s);
  int chunk = (max_context + s - 1) / s;
  chunk = (chunk + DC_KT - 1) / DC_KT * DC_KT;
  p.chunk = chunk;
  p.splits = (max_context + chunk - 1) / chunk;
  return p;
}

}  // namespace attn
}  // namespace qw

using namespace qw;
using namespace qw::attn;

namespace qw {
int launch_attention_prefill_tc(const void* q, const void* k, const void* v, int64_t kv_rows, const int32_t* cu_q,
                                const int32_t* cu_k, const int32_t* seq_base, int n_seqs, int max_seqlen_q, int nh,
                                int nkv, float scale, void* out, cudaStream_t st, const KvPages& pages);
}  // namespace qw

extern "C" int qw_attention_prefill(const void* q, const void* k, const void* v, int64_t kv_rows,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, const int32_t* seq_base,
                                    int n_seqs, int max_seqlen_q, int n_heads, int n_kv_heads, int head_dim,
                                    float scale, void* out, int dtype, void* stream) {
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_attention_prefill: dtype %d", dtype);
  if (n_seqs < 0 || max_seqlen_q < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill: bad sizes");
  if (n_heads % n_kv_heads) return set_error(QW_ERR_SHAPE, "qw_attention_prefill: nh %% nkv != 0");
  if (!(head_dim == 128 && dtype == QW_BF16) && head_dim > 64)
    return set_error(QW_ERR_SHAPE, "qw_attention_prefill: head_dim %d (bf16 needs 128 or <= 64, f32 <= 64)", head_dim);
  if (n_seqs == 0 || max_seqlen_q == 0) return QW_OK;
  if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill: null pointer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == QW_BF16 && head_dim == 128) {
    if (kv_rows <= 0 || (reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) % 16)
      return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill: kv_rows must be > 0 and k, v 16-byte aligned");
    return launch_attention_prefill_tc(q, k, v, kv_rows, cu_seqlens_q, cu_seqlens_k, seq_base, n_seqs, max_seqlen_q,
                                       n_heads, n_kv_heads, scale, out, st, KvPages{nullptr, 0, 0});
  }
  if (dtype == QW_BF16)
    return launch_attn_small<bf16>(q, k, v, cu_seqlens_q, cu_seqlens_k, seq_base, nullptr, n_seqs, max_seqlen_q,
                                   n_heads, n_kv_heads, head_dim, scale, out, st);
  return launch_attn_small<float>(q, k, v, cu_seqlens_q, cu_seqlens_k, seq_base, nullptr, n_seqs, max_seqlen_q,
                                  n_heads, n_kv_heads, head_dim, scale, out, st);
}

// SM count of the current device; 152 (GB300) when no device can be queried,
// which only happens on a host checking arguments without launching.
static int device_sms() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  std::lock_guard<std::mutex> lk(mu);
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

// The persistent decode kernel's workspace: completion counters, then one
// (m, l) and one o per (slot, q head of the group) for the W + B * nkv slots.
// G * W never exceeds 8 * SMs (at most two CTAs per SM of the ~100 KB ring
// for G <= 4, one for G = 8), which bounds it without knowing nkv.
static size_t decode_tc_workspace_bound(int B, int n_heads) {
  return kCounterBytes + (size_t(8) * device_sms() + size_t(B) * n_heads) * (DC_HD + 2) * sizeof(float);
}

extern "C" size_t qw_attention_decode_workspace_size(int B, int max_context, int n_heads, int head_dim) {
  if (B <= 0 || max_context < 0 || n_heads <= 0 || head_dim != 128) return 0;
  size_t need = decode_tc_workspace_bound(B, n_heads);   // bf16
  const DecodePlan p = decode_plan(B, max_context, 0);   // f32 split plan
  if (p.splits > 1) {
    const size_t f32 = kCounterBytes + size_t(B) * n_heads * p.splits * (size_t(head_dim) + 2) * sizeof(float);
    need = need > f32 ? need : f32;
  }
  return need;
}

// Resident CTAs per SM of attn_decode_tc_kernel<G> (its shared memory sets it); set up once.
template <int G>
static int decode_tc_ctas_per_sm(int* out) {
  static std::mutex mu;
  static int v = 0;
  std::lock_guard<std::mutex> lk(mu);
  if (v == 0) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(dt_smem<G>()));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_tc_kernel<G>, DT_THREADS, dt_smem<G>());
    if (e != cudaSuccess || n <= 0)
      return set_error(QW_ERR_CUDA, "decode attention occupancy: %s", cudaGetErrorString(e));
    v = n;
  }
  *out = v;
  return QW_OK;
}

template <int G>
static int launch_decode_tc(const void* q, const void* kc, const void* vc, const int32_t* cl, const int32_t* sb,
                            int B, int nh, int nkv, int64_t num_slots, int max_context, float sl2, void* ws,
                            size_t ws_bytes, int history_ready, void* out, cudaStream_t st,
                            const DecodeRope& rp = DecodeRope{}, const KvPages& pages = KvPages{nullptr, 0, 0}) {
  int per_sm = 0;
  int rc = decode_tc_ctas_per_sm<G>(&per_sm);
  if (rc) return rc;
  // One wave.  With fewer pairs than resident slots, each pair is cut into S
  // equal key chunks (T padded to S * per), so the CTAs of one sequence's kv
  // heads stream the same key rows side by side; otherwise the pairs' tiles
  // are dealt out evenly.  Either way a CTA gets at least two tiles.
  int T = max_context > 0 ? (max_context + DT_KT - 1) / DT_KT : 1;   // max_context 0: empty sequences only
  const int64_t n_pairs = int64_t(B) * nkv;
  int64_t slots_sm = int64_t(device_sms()) * per_sm;
  if (slots_sm > 8 * device_sms() / G) slots_sm = 8 * device_sms() / G;   // keeps the workspace bound
  int64_t per, W;
  if (n_pairs <= slots_sm) {
    int64_t S = slots_sm / n_pairs;
    if (S > (T + 1) / 2) S = (T + 1) / 2;
    if (S < 1) S = 1;
    per = (T + S - 1) / S;
    S = (T + per - 1) / per;
    T = int(S * per);
    W = n_pairs * S;
  } else {
    const int64_t tiles = n_pairs * T;
    W = slots_sm;
    if ((tiles + 1) / 2 < W) W = (tiles + 1) / 2;
    if (W < 1) W = 1;
    per = (tiles + W - 1) / W;
    W = (tiles + per - 1) / per;   // CTAs that get tiles
  }
  const size_t slots = size_t(W) + size_t(n_pairs);
  const size_t need = kCounterBytes + slots * G * (DC_HD + 2) * sizeof(float);
  if (!ws || ws_bytes < need) return set_error(QW_ERR_WORKSPACE, "qw_attention_decode: workspace of %zu bytes needed", need);
  unsigned int* cnt = static_cast<unsigned int*>(ws);
  float* wml = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kCounterBytes);
  float* wo = wml + slots * G * 2;
  CUtensorMap mk, mv;
  const uint64_t dims[3] = {uint64_t(DC_HD), uint64_t(nkv), uint64_t(num_slots)};
  const uint64_t strides[2] = {uint64_t(DC_HD) * 2, uint64_t(nkv) * DC_HD * 2};
  const uint32_t box[3] = {64u, 1u, uint32_t(DT_KT)};
  rc = make_tensor_map(&mk, kc, 3, dims, strides, box);
  if (rc) return rc;
  rc = make_tensor_map(&mv, vc, 3, dims, strides, box);
  if (rc) return rc;
  launch_pdl(attn_decode_tc_kernel<G>, dim3(unsigned(W)), DT_THREADS, dt_smem<G>(), st, mk, mv,
             static_cast<const bf16*>(q), cl, sb, nh, nkv, int(n_pairs), T, int(per), sl2, history_ready, wo, wml,
             cnt, static_cast<bf16*>(out), rp, pages);
  return check_launch("attn_decode_tc_kernel");
}

template <typename T, int G>
static int launch_decode(const void* q, const void* kc, const void* vc, const int32_t* cl, const int32_t* sb, int B,
                         int nh, int nkv, float sl2, const DecodePlan& p, float* wo, float* wml, unsigned int* cnt,
                         void* out, cudaStream_t st) {
  constexpr size_t sm = decode_smem<T>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  dim3 grid(unsigned(p.splits), unsigned(nkv), unsigned(B));
  launch_pdl(attn_decode_kernel<T, G>, grid, DC_THREADS, sm, st, static_cast<const T*>(q), static_cast<const T*>(kc),
                                                         static_cast<const T*>(vc), cl, sb, nh, nkv, sl2, p.chunk,
                                                         p.splits, wo, wml, cnt, static_cast<T*>(out));
  return check_launch("attn_decode_kernel");
}

extern "C" int qw_attention_decode(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                                   const int32_t* context_lens, const int32_t* seq_base, int B, int max_context,
                                   int n_heads, int n_kv_heads, int head_dim, float scale, void* out, void* workspace,
                                   size_t workspace_bytes, int dtype, int flags, void* stream) {
  if (flags & ~QW_DECODE_HISTORY_READY) return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode: flags %d", flags);
  if (dtype != QW_BF16 && dtype != QW_F32) return set_error(QW_ERR_DTYPE, "qw_attention_decode: dtype %d", dtype);
  if (B < 0 || max_context < 0 || n_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || num_slots < 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode: bad sizes");
  if (n_heads % n_kv_heads || (head_dim != 128 && head_dim > 64))
    return set_error(QW_ERR_SHAPE, "qw_attention_decode: needs nh %% nkv == 0 and head_dim 128 or <= 64");
  const int G = n_heads / n_kv_heads;
  if (head_dim == 128 && G != 1 && G != 2 && G != 4 && G != 8)
    return set_error(QW_ERR_SHAPE, "qw_attention_decode: group %d", G);
  if (B == 0) return QW_OK;
  if (!q || !k_cache || !v_cache || !context_lens || !seq_base || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode: null pointer");
  if (head_dim != 128) {
    cudaStream_t st0 = static_cast<cudaStream_t>(stream);
    return dtype == QW_BF16
               ? launch_attn_small<bf16>(q, k_cache, v_cache, nullptr, nullptr, seq_base, context_lens, B, 1, n_heads,
                                         n_kv_heads, head_dim, scale, out, st0)
               : launch_attn_small<float>(q, k_cache, v_cache, nullptr, nullptr, seq_base, context_lens, B, 1,
                                          n_heads, n_kv_heads, head_dim, scale, out, st0);
  }
  if (size_t(B) * n_kv_heads * sizeof(unsigned int) > kCounterBytes)
    return set_error(QW_ERR_SHAPE, "qw_attention_decode: %d sequences x %d kv heads exceed the counter area", B,
                     n_kv_heads);
  const float sl2 = scale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == QW_BF16) {
    const size_t bound = decode_tc_workspace_bound(B, n_heads);
    if (!workspace || workspace_bytes < bound)
      return set_error(QW_ERR_WORKSPACE, "qw_attention_decode: workspace of %zu bytes needed", bound);
    if (reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
      return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode: caches must be 16-byte aligned");
    switch (G) {
      case 1: return launch_decode_tc<1>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, num_slots,
                                         max_context, sl2, workspace, workspace_bytes, flags & QW_DECODE_HISTORY_READY,
                                         out, st);
      case 2: return launch_decode_tc<2>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, num_slots,
                                         max_context, sl2, workspace, workspace_bytes, flags & QW_DECODE_HISTORY_READY,
                                         out, st);
      case 4: return launch_decode_tc<4>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, num_slots,
                                         max_context, sl2, workspace, workspace_bytes, flags & QW_DECODE_HISTORY_READY,
                                         out, st);
      default: return launch_decode_tc<8>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads,
                                          num_slots, max_context, sl2, workspace, workspace_bytes,
                                          flags & QW_DECODE_HISTORY_READY, out, st);
    }
  }
  const DecodePlan p = decode_plan(B, max_context, n_kv_heads);
  const size_t need = p.splits > 1 ? kCounterBytes + size_t(B) * n_heads * p.splits * (DC_HD + 2) * sizeof(float) : 0;
  if (need && (!workspace || workspace_bytes < need))
    return set_error(QW_ERR_WORKSPACE, "qw_attention_decode: workspace of %zu bytes needed", need);
  unsigned int* cnt = need ? static_cast<unsigned int*>(workspace) : nullptr;
  float* wml = need ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + kCounterBytes) : nullptr;
  float* wo = wml ? wml + size_t(B) * n_heads * p.splits * 2 : nullptr;
#define QW_DEC(TT)                                                                                                   \
  switch (G) {                                                                                                       \
    case 1: return launch_decode<TT, 1>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, sl2, p, \
                                        wo, wml, cnt, out, st);                                                           \
    case 2: return launch_decode<TT, 2>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, sl2, p, \
                                        wo, wml, cnt, out, st);                                                           \
    case 4: return launch_decode<TT, 4>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, sl2, p, \
                                        wo, wml, cnt, out, st);                                                           \
    default: return launch_decode<TT, 8>(q, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads, sl2,  \
                                         p, wo, wml, cnt, out, st);                                                       \
  }
  QW_DEC(float)
#undef QW_DEC
}

extern "C" int qw_attention_decode_rope(const void* qkv, int n_heads, int n_kv_heads, int head_dim, int tp,
                                        const int64_t* positions, const float* cos_sin, int64_t max_position,
                                        const void* q_gamma, const void* k_gamma, float eps,
                                        const int64_t* slot_mapping, void* k_cache, void* v_cache, int64_t num_slots,
                                        int32_t* err_count, const int32_t* context_lens, const int32_t* seq_base,
                                        int B, int max_context, float scale, void* out, void* workspace,
                                        size_t workspace_bytes, int dtype, int flags, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_attention_decode_rope: bf16 only");
  if (flags & ~QW_DECODE_HISTORY_READY)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_rope: flags %d", flags);
  if (B < 0 || max_context < 0 || n_heads <= 0 || n_kv_heads <= 0 || tp <= 0 || num_slots < 0 || max_position <= 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_rope: bad sizes");
  const int G = n_kv_heads > 0 ? n_heads / n_kv_heads : 0;
  if (head_dim != 128 || n_heads % n_kv_heads || n_heads % tp || n_kv_heads % tp ||
      (G != 1 && G != 2 && G != 4 && G != 8))
    return set_error(QW_ERR_SHAPE,
                     "qw_attention_decode_rope: needs head_dim 128, nh %% nkv == 0 with group 1/2/4/8, tp | nh, nkv");
  if (B == 0) return QW_OK;
  if (!qkv || !positions || !cos_sin || !q_gamma || !k_gamma || !slot_mapping || !k_cache || !v_cache ||
      !context_lens || !seq_base || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_rope: null pointer");
  if (reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_rope: caches must be 16-byte aligned");
  if (size_t(B) * n_kv_heads * sizeof(unsigned int) > kCounterBytes)
    return set_error(QW_ERR_SHAPE, "qw_attention_decode_rope: %d sequences x %d kv heads exceed the counter area",
                     B, n_kv_heads);
  const size_t bound = decode_tc_workspace_bound(B, n_heads);
  if (!workspace || workspace_bytes < bound)
    return set_error(QW_ERR_WORKSPACE, "qw_attention_decode_rope: workspace of %zu bytes needed", bound);
  DecodeRope rp;
  rp.qkv = static_cast<const bf16*>(qkv);
  rp.positions = positions;
  rp.slots = slot_mapping;
  rp.cos_sin = cos_sin;
  rp.max_pos = max_position;
  rp.q_gamma = static_cast<const bf16*>(q_gamma);
  rp.k_gamma = static_cast<const bf16*>(k_gamma);
  rp.eps = eps;
  rp.tp = tp;
  rp.err = err_count;
  rp.k_cache = static_cast<bf16*>(k_cache);
  rp.v_cache = static_cast<bf16*>(v_cache);
  rp.num_slots = num_slots;
  const float sl2 = scale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int hr = flags & QW_DECODE_HISTORY_READY;
  switch (G) {
    case 1: return launch_decode_tc<1>(nullptr, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads,
                                       num_slots, max_context, sl2, workspace, workspace_bytes, hr, out, st, rp);
    case 2: return launch_decode_tc<2>(nullptr, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads,
                                       num_slots, max_context, sl2, workspace, workspace_bytes, hr, out, st, rp);
    case 4: return launch_decode_tc<4>(nullptr, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads,
                                       num_slots, max_context, sl2, workspace, workspace_bytes, hr, out, st, rp);
    default: return launch_decode_tc<8>(nullptr, k_cache, v_cache, context_lens, seq_base, B, n_heads, n_kv_heads,
                                        num_slots, max_context, sl2, workspace, workspace_bytes, hr, out, st, rp);
  }
}

// Paged KV cache ([SK] §7.2 with a block table): the bf16 head_dim-128 kernels,
// rows found through the block table instead of a contiguous base.
static int check_pages(const char* who, const int32_t* table, int max_blocks, int block_size, int tile) {
  if (!table) return set_error(QW_ERR_INVALID_ARG, "%s: null block table", who);
  if (max_blocks <= 0 || block_size <= 0 || block_size % tile)
    return set_error(QW_ERR_SHAPE, "%s: block_size %d must be a positive multiple of %d", who, block_size, tile);
  return QW_OK;
}

extern "C" int qw_attention_decode_paged(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                                         const int32_t* context_lens, const int32_t* block_table, int max_blocks,
                                         int block_size, int B, int max_context, int n_heads, int n_kv_heads,
                                         int head_dim, float scale, void* out, void* workspace,
                                         size_t workspace_bytes, int dtype, int flags, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_attention_decode_paged: bf16 only");
  if (flags & ~QW_DECODE_HISTORY_READY)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_paged: flags %d", flags);
  if (B < 0 || max_context < 0 || n_heads <= 0 || n_kv_heads <= 0 || num_slots < 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_paged: bad sizes");
  const int G = n_heads / n_kv_heads;
  if (head_dim != 128 || n_heads % n_kv_heads || (G != 1 && G != 2 && G != 4 && G != 8))
    return set_error(QW_ERR_SHAPE, "qw_attention_decode_paged: needs head_dim 128 and group 1/2/4/8");
  int rc = check_pages("qw_attention_decode_paged", block_table, max_blocks, block_size, DT_KT);
  if (rc) return rc;
  if (int64_t(max_context) > int64_t(max_blocks) * block_size)
    return set_error(QW_ERR_SHAPE, "qw_attention_decode_paged: max_context %d > max_blocks x block_size", max_context);
  if (B == 0) return QW_OK;
  if (!q || !k_cache || !v_cache || !context_lens || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_paged: null pointer");
  if (reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_decode_paged: caches must be 16-byte aligned");
  if (size_t(B) * n_kv_heads * sizeof(unsigned int) > kCounterBytes)
    return set_error(QW_ERR_SHAPE, "qw_attention_decode_paged: %d sequences x %d kv heads exceed the counter area", B,
                     n_kv_heads);
  const size_t bound = decode_tc_workspace_bound(B, n_heads);
  if (!workspace || workspace_bytes < bound)
    return set_error(QW_ERR_WORKSPACE, "qw_attention_decode_paged: workspace of %zu bytes needed", bound);
  const KvPages pages{block_table, max_blocks, block_size};
  const float sl2 = scale * kLog2e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int hr = flags & QW_DECODE_HISTORY_READY;
  switch (G) {
    case 1: return launch_decode_tc<1>(q, k_cache, v_cache, context_lens, nullptr, B, n_heads, n_kv_heads, num_slots,
                                       max_context, sl2, workspace, workspace_bytes, hr, out, st, DecodeRope{}, pages);
    case 2: return launch_decode_tc<2>(q, k_cache, v_cache, context_lens, nullptr, B, n_heads, n_kv_heads, num_slots,
                                       max_context, sl2, workspace, workspace_bytes, hr, out, st, DecodeRope{}, pages);
    case 4: return launch_decode_tc<4>(q, k_cache, v_cache, context_lens, nullptr, B, n_heads, n_kv_heads, num_slots,
                                       max_context, sl2, workspace, workspace_bytes, hr, out, st, DecodeRope{}, pages);
    default: return launch_decode_tc<8>(q, k_cache, v_cache, context_lens, nullptr, B, n_heads, n_kv_heads,
                                        num_slots, max_context, sl2, workspace, workspace_bytes, hr, out, st,
                                        DecodeRope{}, pages);
  }
}

extern "C" int qw_attention_prefill_paged(const void* q, const void* k_cache, const void* v_cache, int64_t num_slots,
                                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                          const int32_t* block_table, int max_blocks, int block_size, int n_seqs,
                                          int max_seqlen_q, int n_heads, int n_kv_heads, int head_dim, float scale,
                                          void* out, int dtype, void* stream) {
  if (dtype != QW_BF16) return set_error(QW_ERR_DTYPE, "qw_attention_prefill_paged: bf16 only");
  if (n_seqs < 0 || max_seqlen_q < 0 || n_heads <= 0 || n_kv_heads <= 0 || num_slots <= 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill_paged: bad sizes");
  if (head_dim != 128 || n_heads % n_kv_heads)
    return set_error(QW_ERR_SHAPE, "qw_attention_prefill_paged: needs head_dim 128 and nh %% nkv == 0");
  int rc = check_pages("qw_attention_prefill_paged", block_table, max_blocks, block_size, 128);
  if (rc) return rc;
  if (n_seqs == 0 || max_seqlen_q == 0) return QW_OK;
  if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !out)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill_paged: null pointer");
  if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_attention_prefill_paged: caches must be 16-byte aligned");
  return launch_attention_prefill_tc(q, k_cache, v_cache, num_slots, cu_seqlens_q, cu_seqlens_k, nullptr, n_seqs,
                                     max_seqlen_q, n_heads, n_kv_heads, scale, out, static_cast<cudaStream_t>(stream),
                                     KvPages{block_table, max_blocks, block_size});
}

// ===========================================================================
// Decode attention without any device allocation by the caller.
//
// Some callers cannot hand this library a workspace: a plugin inside a host
// framework that owns the device allocator and passes in only its input and
// output pointers, or a serving loop that plans all device memory at
// start-up and allows no allocation afterwards.  For them the split-KV
// partial results live in one fixed array in this library's device image.
// ===========================================================================
namespace qw {
namespace attn {

constexpr size_t kStaticScratchBytes = size_t(2) << 20;   // 2 MiB on every GPU that loads the library
static __device__ __align__(256) float g_decode_scratch[kStaticScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device, looked up once per
// device (host code only sees a host-side stand-in for the array's name).
static int decode_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(QW_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || p == nullptr)
      return set_error(QW_ERR_CUDA, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QW_OK;
}

}  // namespace attn
}  // namespace qw

extern "C" size_t qw_attention_decode_static_scratch_bytes(void) { return qw::attn::kStaticScratchBytes; }

extern "C" int qw_attention_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                          int64_t num_slots, const int32_t* context_lens, const int32_t* seq_base, int B,
                                          int max_context, int n_heads, int n_kv_heads, int head_dim, float scale,
                                          void* out, int dtype, void* stream) {
  const size_t need = qw_attention_decode_workspace_size(B, max_context, n_heads, head_dim);
  if (need > qw::attn::kStaticScratchBytes)
    return set_error(QW_ERR_WORKSPACE,
                     "qw_attention_decode_static: this batch needs %zu bytes of split-KV scratch but the fixed "
                     "array holds %zu; pass a workspace to qw_attention_decode instead",
                     need, qw::attn::kStaticScratchBytes);
  void* ws = nullptr;
  if (need > 0) {
    const int rc = qw::attn::decode_scratch_address(&ws);
    if (rc != QW_OK) return rc;
  }
  return qw_attention_decode(q, k_cache, v_cache, num_slots, context_lens, seq_base, B, max_context, n_heads, n_kv_heads,
                             head_dim, scale, out, ws, need > 0 ? qw::attn::kStaticScratchBytes : 0, dtype, 0, stream);
}

namespace qw {
unsigned int take_attn_timeouts() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, attn::g_attn_timeout, sizeof(v));
  if (v) cudaMemcpyToSymbol(attn::g_attn_timeout, &z, sizeof(z));
  return v;
}
}  // namespace qw
