// One decode step of every decoder layer as a single persistent kernel
// (Qwen3DecoderLayer.forward x n_layers, [SK] §1, §8), for batches of at
// most 16 new tokens, where each layer's work is too small to fill the GPU
// one operator at a time.
//
// One CTA per SM (a cooperative launch, so all CTAs are resident), 9 warps:
//   warp 0     weight producer: streams this CTA's share of every weight
//              matrix, layer after layer, through a shared-memory ring.  A
//              copy request is one whole weight row (2-3 KB): the bulk-copy
//              engine costs about the same per request whatever its size,
//              and requests of 2 KB or more reach full HBM bandwidth.  It
//              never waits for activations, so weights stream ahead across
//              stage boundaries.
//   warps 1-4  attention consumers; all of warps 1-8 run the GEMVs and norms
//   warp 5     attention producer during the attention stage
// Per layer, separated by grid-wide barriers:
//   A  input RMSNorm of (h + residual), recomputed in every CTA for all
//      tokens into shared memory; CTA 0 writes the new residual
//   B  QKV GEMV (column layout)
//   C  attention over (sequence, kv head, key chunk) items claimed
//      dynamically: the producer warp claims items, stores the new token's
//      k (QK-RMSNorm + RoPE) and v to the cache for the item that covers it,
//      and keeps a 3-stage ring of 64-key K/V tiles full (TMA, 128-byte
//      swizzle); it starts on the cached history before the barrier that
//      publishes this step's QKV.  The consumer warps normalise and rotate
//      the item's q heads, run the online softmax with warp-level MMAs, and
//      the last chunk of a (sequence, kv head) merges all chunks.
//   D  o_proj GEMV (row layout: the tp shards' partial sums are added)
//   E  post-attention RMSNorm as in A, then gate_up GEMV + SiluAndMul
//   F  down GEMV (row layout)
// then the final RMSNorm.  Each CTA of a GEMV owns a contiguous run of
// about N / #SMs outputs (equal weight bytes per SM to within one row); a
// unit is up to 12 of those rows (6 gate + 6 up rows for gate_up) over one
// shard's K.  Results do not depend on timing: every sum has a fixed order.
//
// Every wait is bounded (2 s of %globaltimer).  A timeout sets an error
// word that every other wait checks, so the kernel then runs to its end
// without waiting; the host reports it through qw_device_error.
#include <cuda.h>
#include <math.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "tc_common.cuh"

namespace qw {
namespace dstep {

__device__ unsigned int g_dstep_error = 0;

constexpr int HD = 128;
constexpr int MAXL = 64;                        // layers per call
constexpr int NCW = 8;                          // compute warps (1..8)
constexpr int THREADS = (NCW + 1) * 32;
constexpr int MAXB = 16;
constexpr int SLOT = 12 * (2048 + 64);          // weight ring slot: 12 rows of 1024 bf16 (padded)
constexpr int ATT_KT = 64;                      // keys per attention tile
constexpr uint32_t ATT_BOX = ATT_KT * 64 * 2;   // 64 keys x 64 dims (one 128-byte-swizzled box)
constexpr uint32_t ATT_STAGE = 4 * ATT_BOX;     // K dims 0-63, K 64-127, V 0-63, V 64-127
constexpr int ATT_STAGES = 3;
constexpr int ITEMQ = 4;                        // attention item queue depth
constexpr int YPAD = 32;                        // activation row padding (elements)
constexpr uint64_t kTimeoutNs = 2000000000ull;
enum { G_QKV = 0, G_O = 1, G_GU = 2, G_DOWN = 3 };

// one layer's parameters; the layout of qw_decode_layer in include/qw.h
struct LayerPtrs {
  const bf16* input_ln;
  const bf16* qkv;       // [tp * (nh/tp + 2 nkv/tp) * hd, H]
  const bf16* q_norm;
  const bf16* k_norm;
  const bf16* o;         // [tp, H, nh/tp * hd]
  const bf16* post_ln;
  const bf16* gate_up;   // [tp * 2 I/tp, H]
  const bf16* down;      // [tp, H, I/tp]
  bf16* k_cache;         // [num_slots, nkv, hd]
  bf16* v_cache;
};

struct Params {
  CUtensorMap kmap[MAXL];       // K / V cache of each layer: {hd, nkv, num_slots}, box {64, 1, 64}
  CUtensorMap vmap[MAXL];
  LayerPtrs layers[MAXL];
  int n_layers, B, H, nh, nkv, I, tp;
  const bf16* x;
  const bf16* final_ln;
  bf16* out;
  const int64_t* positions;
  const int64_t* slots;
  const int32_t* ctx_lens;
  const int32_t* seq_base;
  const float* cos_sin;
  int64_t max_pos, num_slots;
  float eps, scale_log2;
  int att_chunk, att_splits;
  int ring;                     // weight ring slots
  int red_units;                // o_proj / down units of one CTA (partial tiles in shared memory)
  uint32_t union_bytes;         // attention ring / activations staging region
  // workspace
  unsigned long long* bar;
  unsigned int* err;
  unsigned int* work;           // [n_layers] attention item counters
  unsigned int* cnt_att;        // [B * nkv]
  int32_t* err_count;           // bad positions / slots (may be null)
  float* att_o;                 // [B, nh, splits, hd]
  float* att_ml;                // [B, nh, splits, 2]
  bf16* qkv_buf;                // [B, qkv width]
  bf16* attn_buf;               // [B, nh * hd]
  bf16* act_buf;                // [B, I]
  bf16* h_buf;                  // [B, H]
  bf16* res_buf;                // [2, B, H]
};

// ---------------------------------------------------------------------------
// GEMV geometry (identical in the weight producer and the consumers)
// ---------------------------------------------------------------------------
struct Gemv {
  int n_out;    // outputs (rows; gate_up: SiluAndMul columns)
  int K;        // input width (all shards)
  int kseg;     // k values per row request: one shard's K (row layouts) or K
  int nseg;     // requests per row: tp (o_proj, down) or 1
  int R;        // outputs per unit
  int stride;   // bytes per staged row
  int o0, o1;   // this CTA's outputs
  int tiles, units;
};
__host__ __device__ __forceinline__ Gemv gemv_geom(int which, int H, int nh, int nkv, int I, int tp, int cta,
                                                   int nctas) {
  Gemv g;
  const int qkvw = (nh + 2 * nkv) * HD;
  switch (which) {
    case G_QKV: g.n_out = qkvw; g.K = H; g.nseg = 1; break;
    case G_O: g.n_out = H; g.K = nh * HD; g.nseg = tp; break;
    case G_GU: g.n_out = I; g.K = H; g.nseg = 1; break;
    default: g.n_out = H; g.K = I; g.nseg = tp; break;
  }
  g.kseg = g.K / g.nseg;
  g.stride = g.kseg * 2 + 64;   // (stride / 16) % 8 == 4: conflict-free 16-byte fragment reads
  g.R = which == G_GU ? (SLOT / (2 * g.stride) < 8 ? SLOT / (2 * g.stride) : 8)
                      : (SLOT / g.stride < 16 ? SLOT / g.stride : 16);
  g.o0 = int(int64_t(g.n_out) * cta / nctas);
  g.o1 = int(int64_t(g.n_out) * (cta + 1) / nctas);
  g.tiles = g.R > 0 ? (g.o1 - g.o0 + g.R - 1) / g.R : 0;
  g.units = g.tiles * g.nseg;
  return g;
}
__device__ __forceinline__ Gemv gemv_of(const Params& p, int which) {
  return gemv_geom(which, p.H, p.nh, p.nkv, p.I, p.tp, blockIdx.x, gridDim.x);
}

__device__ __forceinline__ bool failed(const Params& p) {
  return *reinterpret_cast<volatile unsigned int*>(p.err) != 0u;
}
__device__ __forceinline__ void raise(const Params& p, unsigned int code) {
  atomicOr(p.err, code);
  atomicOr(&g_dstep_error, code);
}
__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* a) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
  return v;
}
// bounded mbarrier wait that gives up at once after any failure
__device__ __forceinline__ bool bwait(const Params& p, uint32_t bar, uint32_t parity, unsigned int code) {
  if (tcx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = tcx::globaltimer();
  while (true) {
    if (tcx::mbar_try_wait(bar, parity)) return true;
    if (failed(p)) return false;
    if (tcx::globaltimer() - t0 > kTimeoutNs) {
      raise(p, code);
      return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint4 ldcg16(const void* p) { return __ldcg(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ void prefetch_l1(const void* p) { asm volatile("prefetch.global.L1 [%0];" ::"l"(p)); }
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
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
__device__ __forceinline__ float silu_mul(float g, float u) {
  g = round_t<bf16>(g);   // gate_up is a model-dtype tensor before SiluAndMul
  u = round_t<bf16>(u);
  return g / (1.0f + expf(-g)) * u;
}
// byte offset of (key row r, 16-byte chunk c16 of the 128 dims) in a K or V tile
__device__ __forceinline__ uint32_t kv_off(int r, int c16) {
  return uint32_t(c16 >> 3) * ATT_BOX + uint32_t(r) * 128u + uint32_t(((c16 & 7) ^ (r & 7)) * 16);
}

// ---------------------------------------------------------------------------
// grid-wide barrier over the compute warps of every CTA.  A 64-bit arrival
// counter only grows and is a multiple of gridDim.x between launches; each
// CTA reads it once at start (rounded down to that multiple: no barrier of
// this launch can complete before every CTA has arrived at it) and barrier k
// of the launch waits for base + (k+1) * gridDim.x arrivals.  The release
// add also publishes every write the CTA made before its named barrier.
// ---------------------------------------------------------------------------
__device__ void grid_arrive(const Params& p, unsigned long long& target) {
  named_sync(1, NCW * 32);
  if (threadIdx.x == 32) {
    target += gridDim.x;
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(p.bar) : "memory");
  }
}
__device__ void grid_wait(const Params& p, unsigned long long target) {
  if (threadIdx.x == 32) {
    const uint64_t t0 = tcx::globaltimer();
    while (static_cast<long long>(ld_acquire_u64(p.bar) - target) < 0) {
      if (failed(p)) break;
      if (tcx::globaltimer() - t0 > kTimeoutNs) {
        raise(p, 1u << 0);
        break;
      }
    }
  }
  named_sync(1, NCW * 32);
}
__device__ __forceinline__ void grid_sync(const Params& p, unsigned long long& target) {
  grid_arrive(p, target);
  grid_wait(p, target);
}

// ---------------------------------------------------------------------------
// weight rows: output o's row (gate_up: its gate row, or its up row)
// ---------------------------------------------------------------------------
__device__ __forceinline__ const bf16* weight_row(const Params& p, const LayerPtrs& lw, int which, const Gemv& gm,
                                                  int o, int seg, bool up) {
  switch (which) {
    case G_QKV:
      return lw.qkv + int64_t(o) * p.H;
    case G_O:
      return lw.o + (int64_t(seg) * p.H + o) * gm.kseg;
    case G_GU: {
      const int il = p.I / p.tp;
      const int s = o / il, jj = o - s * il;
      return lw.gate_up + (int64_t(s) * 2 * il + (up ? il : 0) + jj) * p.H;
    }
    default:
      return lw.down + (int64_t(seg) * p.H + o) * gm.kseg;
  }
}

// ---------------------------------------------------------------------------
// warp 0: weight producer
// ---------------------------------------------------------------------------
__device__ void producer(const Params& p, uint8_t* wring, uint64_t* wfull, uint64_t* wempty) {
  const int lane = threadIdx.x & 31;
  int64_t pos = 0;
  bool ok = true;
  for (int l = 0; l < p.n_layers && ok; ++l) {
    const LayerPtrs& lw = p.layers[l];
    for (int which = 0; which < 4 && ok; ++which) {
      const Gemv gm = gemv_of(p, which);
      for (int u = 0; u < gm.units; ++u, ++pos) {
        const int slot = int(pos % p.ring);
        if (pos >= p.ring && !bwait(p, smem_u32(wempty + slot), uint32_t((pos / p.ring) - 1) & 1u, 1u << 1)) {
          ok = false;
          break;
        }
        const int t = u / gm.nseg, seg = u % gm.nseg;
        const int n = min(gm.R, gm.o1 - gm.o0 - t * gm.R);   // outputs of this unit
        const int reqs = which == G_GU ? 2 * n : n;
        const uint32_t dst = smem_u32(wring + size_t(slot) * SLOT);
        // the consumers' generic reads of this slot before the async-proxy copies refill it
        tcx::fence_proxy_async();
        if (lane == 0) tcx::mbar_expect_tx(smem_u32(wfull + slot), uint32_t(reqs) * gm.kseg * 2u);
        __syncwarp();
        for (int r = lane; r < reqs; r += 32) {
          const bool up = which == G_GU && r >= n;
          const int j = up ? r - n : r;
          const int srow = up ? gm.R + j : j;
          bulk_g2s(dst + uint32_t(srow * gm.stride), weight_row(p, lw, which, gm, gm.o0 + t * gm.R + j, seg, up),
                   gm.kseg * 2u, smem_u32(wfull + slot));
        }
        __syncwarp();
      }
    }
  }
  // the last copies have landed before the CTA may exit
  for (int64_t q = max(int64_t(0), pos - p.ring); q < pos; ++q)
    bwait(p, smem_u32(wfull + int(q % p.ring)), uint32_t(q / p.ring) & 1u, 1u << 2);
}

// ---------------------------------------------------------------------------
// RMSNorm of (h + residual) for all tokens into shared memory (compute warps)
// ---------------------------------------------------------------------------
__device__ void norm_stage(const Params& p, const bf16* hin, const bf16* res_in, bf16* res_out, const bf16* gamma,
                           bf16* ys) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int ystride = p.H + YPAD;
  constexpr int MAXV = 4;   // 16-byte vectors per lane in flight at once (one pass for H <= 1024)
  const int nv = p.H / 256;
  for (int t = cw; t < p.B; t += NCW) {
    float ss = 0.0f;
    for (int i0 = 0; i0 < nv; i0 += MAXV) {
      uint4 hv[MAXV], rv[MAXV];
#pragma unroll
      for (int i = 0; i < MAXV; ++i)   // every load of the pass in flight before any use
        if (i0 + i < nv) {
          hv[i] = ldcg16(hin + int64_t(t) * p.H + (i0 + i) * 256 + lane * 8);
          if (res_in != nullptr) rv[i] = ldcg16(res_in + int64_t(t) * p.H + (i0 + i) * 256 + lane * 8);
          prefetch_l1(gamma + (i0 + i) * 256 + lane * 8);
        }
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        if (i0 + i >= nv) continue;
        const int k = (i0 + i) * 256 + lane * 8;
        float v[8];
        const bf16* hb = reinterpret_cast<const bf16*>(&hv[i]);
        const bf16* rb = reinterpret_cast<const bf16*>(&rv[i]);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          v[e] = res_in != nullptr ? round_t<bf16>(__bfloat162float(hb[e]) + __bfloat162float(rb[e]))
                                   : __bfloat162float(hb[e]);
        if (res_out != nullptr && blockIdx.x == 0) store16(res_out + int64_t(t) * p.H + k, v);
#pragma unroll
        for (int e = 0; e < 8; ++e) ss += v[e] * v[e];
        store16(ys + t * ystride + k, v);   // the sum, normalised below
      }
    }
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / float(p.H) + p.eps);
    __syncwarp();
    for (int i = 0; i < nv; ++i) {
      const int k = i * 256 + lane * 8;
      float v[8], g[8];
      load16(ys + t * ystride + k, v);
      load16(gamma + k, g);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = (v[e] * inv) * g[e];
      store16(ys + t * ystride + k, v);
    }
  }
  tcx::fence_proxy_async();   // ys shares memory with the attention ring (TMA writes)
  named_sync(1, NCW * 32);
}

// ---------------------------------------------------------------------------
// GEMV stage (compute warps).  Ring slot s is consumed by compute warp
// s % min(ring, 8) for the whole run, so no warp can wait on a slot more
// than one fill ahead of its contents.
//   xs: activations in shared memory, rows of stride xstride elements (the
//   normed y, or o_proj / down inputs staged from global memory here)
// ---------------------------------------------------------------------------
__device__ void gemv_stage(const Params& p, int which, int64_t pos0, uint8_t* wring, uint64_t* wfull,
                           uint64_t* wempty, const bf16* xs, const bf16* xg, bf16* xstage, float* red) {
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const Gemv gm = gemv_of(p, which);
  const int nt = (p.B + 7) / 8;
  int xstride = p.H + YPAD;
  if (xg != nullptr) {
    // activations written by other CTAs: copy all B x K of them into shared
    // memory once (L2 -> shared, no registers), rows padded like ys
    xstride = gm.K + YPAD;
    const int vec = gm.K / 8;
    for (int e = threadIdx.x - 32; e < p.B * vec; e += NCW * 32) {
      const int tok = e / vec, k = (e - tok * vec) * 8;
      cp_async16(smem_u32(xstage + tok * xstride + k), xg + int64_t(tok) * gm.K + k);
    }
    cp_async_commit();
    cp_async_wait<0>();
    named_sync(1, NCW * 32);
    xs = xstage;
  }
  const int ncons = min(p.ring, NCW);
  const bool gu = which == G_GU;
  if (cw < ncons) {
    for (int u = 0; u < gm.units; ++u) {
      const int64_t pos = pos0 + u;
      const int slot = int(pos % p.ring);
      if (slot % ncons != cw) continue;
      const int tl = u / gm.nseg, seg = u % gm.nseg;
      const int n = min(gm.R, gm.o1 - gm.o0 - tl * gm.R);
      // A rows of the MMA: row g <- output g (gate g); row g+8 <- output 8+g (up g)
      const bool okA = g < n;
      const bool okB = gu ? g < n : 8 + g < n;
      const int rowB = gu ? gm.R + g : 8 + g;
      const bool ok = bwait(p, smem_u32(wfull + slot), uint32_t(pos / p.ring) & 1u, 1u << 3);
      const uint8_t* ws = wring + size_t(slot) * SLOT;
      const bf16* xb = xs + seg * gm.kseg;
      // eight independent accumulator chains (a warp-level MMA has a long
      // latency; one chain over 2 * kseg / 32 MMAs would serialise on it);
      // token tiles one after the other (the weights are re-read from
      // shared memory) to keep the accumulators in registers
      for (int m = 0; m < nt; ++m) {
        float acc[8][4];
#pragma unroll
        for (int a = 0; a < 8; ++a) acc[a][0] = acc[a][1] = acc[a][2] = acc[a][3] = 0.0f;
        const int tokx = m * 8 + g;
        if (ok) {
          for (int c0 = 0; c0 < gm.kseg / 32; c0 += 4) {
#pragma unroll
            for (int ci = 0; ci < 4; ++ci) {
              const int kk = 32 * (c0 + ci) + 8 * t;
              const uint4 wa =
                  okA ? *reinterpret_cast<const uint4*>(ws + g * gm.stride + kk * 2) : make_uint4(0, 0, 0, 0);
              const uint4 wb =
                  okB ? *reinterpret_cast<const uint4*>(ws + rowB * gm.stride + kk * 2) : make_uint4(0, 0, 0, 0);
              const uint4 x = tokx < p.B ? *reinterpret_cast<const uint4*>(xb + tokx * xstride + kk)
                                         : make_uint4(0u, 0u, 0u, 0u);
              mma16816(acc[2 * ci], wa.x, wb.x, wa.y, wb.y, x.x, x.y);
              mma16816(acc[2 * ci + 1], wa.z, wb.z, wa.w, wb.w, x.z, x.w);
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[0][e] = ((acc[0][e] + acc[1][e]) + (acc[2][e] + acc[3][e])) +
                        ((acc[4][e] + acc[5][e]) + (acc[6][e] + acc[7][e]));
        }
        // C fragment: rows g, g+8 x tokens 2t, 2t+1 of this n-tile
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = m * 8 + 2 * t + e;
          if (tok >= p.B) continue;
          const float ca = acc[0][e], cb = acc[0][2 + e];
          if (which == G_QKV) {
            bf16* dst = p.qkv_buf + int64_t(tok) * gm.n_out + gm.o0 + tl * gm.R;
            if (okA) dst[g] = __float2bfloat16_rn(ca);
            if (okB) dst[8 + g] = __float2bfloat16_rn(cb);
          } else if (gu) {
            if (okA) p.act_buf[int64_t(tok) * p.I + gm.o0 + tl * gm.R + g] = __float2bfloat16_rn(silu_mul(ca, cb));
          } else {
            // one shard's partial sum: added over the shards below
            float* rt = red + (size_t(tl) * gm.nseg + seg) * 16 * p.B;
            rt[g * p.B + tok] = ca;
            rt[(8 + g) * p.B + tok] = cb;
          }
        }
      }
      __syncwarp();
      if (lane == 0) tcx::mbar_arrive(smem_u32(wempty + slot));
    }
  }
  if (which == G_O || which == G_DOWN) {
    named_sync(1, NCW * 32);
    for (int e = threadIdx.x - 32; e < gm.tiles * 16 * p.B; e += NCW * 32) {
      const int tok = e % p.B, r = (e / p.B) % 16, tl = e / (16 * p.B);
      const int o = gm.o0 + tl * gm.R + r;
      if (r >= gm.R || o >= gm.o1) continue;
      float sum = 0.0f;
      for (int s = 0; s < gm.nseg; ++s) sum += red[(size_t(tl) * gm.nseg + s) * 16 * p.B + r * p.B + tok];
      p.h_buf[int64_t(tok) * p.H + o] = __float2bfloat16_rn(sum);
    }
  }
  if (xg != nullptr) tcx::fence_proxy_async();   // the staging shares memory with the attention ring
}

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
// RMSNorm + RoPE of one head row (128 values at src) by one warp; lane holds
// dims lane, lane+32 (first half) and lane+64, lane+96 (their rotation partners)
__device__ __forceinline__ void norm_rope_head(const Params& p, const bf16* src, const bf16* gamma, int64_t pos,
                                               float (&y)[4]) {
  const int lane = threadIdx.x & 31;
  float x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) x[i] = __bfloat162float(__ldcg(src + lane + 32 * i));   // written by other CTAs
  float ss = x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / float(HD) + p.eps);
  const bool pos_ok = pos >= 0 && pos < p.max_pos;
  const float* cs = p.cos_sin + (pos_ok ? pos : 0) * HD;
  float n[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) n[i] = round_t<bf16>((x[i] * inv) * __bfloat162float(gamma[lane + 32 * i]));
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int d = lane + 32 * i;
    const float c = cs[d], s = cs[64 + d];
    y[i] = pos_ok ? round_t<bf16>(n[i] * c - n[i + 2] * s) : 0.0f;
    y[i + 2] = pos_ok ? round_t<bf16>(n[i + 2] * c + n[i] * s) : 0.0f;
  }
}

constexpr int MERGEQ = 8;   // chunks finished and waiting for the merge warp
struct AttShared {          // attention bookkeeping in shared memory
  uint64_t full[ATT_STAGES], empty[ATT_STAGES];
  uint64_t it_full[ITEMQ], it_empty[ITEMQ];
  uint64_t mq_full[MERGEQ], mq_empty[MERGEQ];
  int item[ITEMQ];
  int merge[MERGEQ];        // (sequence, kv head) of a finished chunk, or -1: end of stage
  // this step's per-token inputs (read once)
  int64_t pos[MAXB], slot[MAXB];
  int ctx[MAXB], base[MAXB];
};
// q of the item in queue slot s: qq + s * G * HD (normed, roped, bf16-valued floats)

struct AttItem {
  int b, g, split, start, end, L;
};
__device__ __forceinline__ AttItem att_item(const Params& p, const AttShared& as, int item) {
  AttItem it;
  it.split = item % p.att_splits;
  const int bg = item / p.att_splits;
  it.b = bg / p.nkv;
  it.g = bg % p.nkv;
  it.L = as.ctx[it.b];
  it.start = it.split * p.att_chunk;
  it.end = min(it.L, it.start + p.att_chunk);
  return it;
}

// attention producer (warp 5): the item queue and the K/V tile ring.  Called
// twice per layer: before the barrier that publishes this step's QKV
// (prefetch: claim the first item and load its cached history without ever
// blocking) and after it (everything else).
struct AttProducer {
  int64_t tile_pos;   // ring position of the next tile (continues across layers)
  int ordinal;        // item queue position (continues across layers)
  int cur, cur_t;     // item being issued and its next tile (-1: none; -2: end marker to publish)
  bool published;     // cur is in the queue
  bool done;
};

template <int G>
__device__ void att_produce(const Params& p, int l, uint8_t* aring, AttShared& as, float* qq, AttProducer& st,
                            bool prefetch) {
  const int lane = threadIdx.x & 31;
  const int n_items = p.B * p.nkv * p.att_splits;
  const CUtensorMap* km = &p.kmap[l];
  const CUtensorMap* vm = &p.vmap[l];
  const LayerPtrs& lw = p.layers[l];
  const int nh_l = p.nh / p.tp, nkv_l = p.nkv / p.tp;
  const int64_t qkvw = int64_t(p.nh + 2 * p.nkv) * HD;
  const int64_t width_r = int64_t(nh_l + 2 * nkv_l) * HD;
  while (!st.done) {
    if (st.cur < 0) {
      // claim the next item; it is published (with its q) once this step's QKV is visible
      const int q = st.ordinal % ITEMQ;
      if (st.ordinal >= ITEMQ) {
        if (prefetch) return;
        if (!bwait(p, smem_u32(&as.it_empty[q]), uint32_t(st.ordinal / ITEMQ - 1) & 1u, 1u << 4)) {
          st.done = true;
          break;
        }
      }
      int item = 0;
      if (lane == 0) item = int(atomicAdd(p.work + l, 1u));
      item = __shfl_sync(0xffffffffu, item, 0);
      st.cur = item < n_items ? item : -1;
      st.cur_t = 0;
      st.published = false;
      if (item >= n_items) {
        if (prefetch) {   // publish the end marker after the barrier
          st.cur = -2;
          return;
        }
        if (lane == 0) {
          as.item[q] = -1;
          tcx::mbar_arrive(smem_u32(&as.it_full[q]));
        }
        __syncwarp();
        ++st.ordinal;
        st.done = true;
        break;
      }
    }
    if (st.cur == -2) {   // end marker claimed before the barrier
      const int q = st.ordinal % ITEMQ;
      if (lane == 0) {
        as.item[q] = -1;
        tcx::mbar_arrive(smem_u32(&as.it_full[q]));
      }
      __syncwarp();
      ++st.ordinal;
      st.done = true;
      break;
    }
    const AttItem it = att_item(p, as, st.cur);
    if (!st.published && !prefetch) {
      // q heads of the item (QK-RMSNorm + RoPE), then publish it
      const int q = st.ordinal % ITEMQ;
      const int64_t pos = as.pos[it.b];
      const bf16* qkv_row = p.qkv_buf + int64_t(it.b) * qkvw + (it.g / nkv_l) * width_r;
      float* qs = qq + q * G * HD;
      for (int j = 0; j < G; ++j) {
        float y[4];
        norm_rope_head(p, qkv_row + int64_t((it.g * G + j) % nh_l) * HD, lw.q_norm, pos, y);
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[j * HD + lane + 32 * i] = y[i];
      }
      __syncwarp();
      if (lane == 0) {
        as.item[q] = st.cur;
        tcx::mbar_arrive(smem_u32(&as.it_full[q]));   // release: the q writes above are visible
      }
      __syncwarp();
      ++st.ordinal;
      st.published = true;
    }
    const int n_t = it.start < it.end ? (it.end - it.start + ATT_KT - 1) / ATT_KT : 0;
    const bool has_new = it.start < it.end && it.end == it.L;   // holds this step's key (position L - 1)
    if (st.cur_t < n_t) {
      if (has_new && st.cur_t == n_t - 1) {
        if (prefetch) return;   // this step's k/v are published by the QKV barrier
        // store the new token's k (normed, roped) and v before loading the tile that holds them
        const int64_t pos = as.pos[it.b];
        const int64_t slot = as.slot[it.b];
        const bool pos_ok = pos >= 0 && pos < p.max_pos;
        if (slot != -1) {
          if (slot < 0 || slot >= p.num_slots || !pos_ok) {
            if (lane == 0 && p.err_count != nullptr && (slot < 0 || slot >= p.num_slots)) atomicAdd(p.err_count, 1);
          } else {
            const bf16* krow = p.qkv_buf + int64_t(it.b) * qkvw + (it.g / nkv_l) * width_r +
                               int64_t(nh_l + it.g % nkv_l) * HD;
            float y[4];
            norm_rope_head(p, krow, lw.k_norm, pos, y);
            bf16* kd = lw.k_cache + (slot * p.nkv + it.g) * int64_t(HD);
            bf16* vd = lw.v_cache + (slot * p.nkv + it.g) * int64_t(HD);
            const bf16* vrow = krow + int64_t(nkv_l) * HD;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              kd[lane + 32 * i] = __float2bfloat16_rn(y[i]);
              vd[lane + 32 * i] = __ldcg(vrow + lane + 32 * i);
            }
          }
        }
        __threadfence();
        asm volatile("fence.proxy.async.global;" ::: "memory");   // visible to the tensor copies below
        __syncwarp();
      }
      const int stg = int(st.tile_pos % ATT_STAGES);
      if (st.tile_pos >= ATT_STAGES) {
        const uint32_t par = uint32_t(st.tile_pos / ATT_STAGES - 1) & 1u;
        if (prefetch) {
          if (!tcx::mbar_try_wait(smem_u32(&as.empty[stg]), par)) return;   // never block before the barrier
        } else if (!bwait(p, smem_u32(&as.empty[stg]), par, 1u << 5)) {
          st.done = true;
          break;
        }
      }
      if (lane == 0) {
        // generic reads of this stage (the consumers' ldmatrix, or the norm and
        // GEMV stages that share the region) before the async-proxy copies
        tcx::fence_proxy_async();
        const uint32_t dst = smem_u32(aring + size_t(stg) * ATT_STAGE);
        const uint32_t fb = smem_u32(&as.full[stg]);
        const int z = as.base[it.b] + it.start + st.cur_t * ATT_KT;
        tcx::mbar_expect_tx(fb, ATT_STAGE);
        tcx::tma_load_3d(dst, km, fb, 0, it.g, z);
        tcx::tma_load_3d(dst + ATT_BOX, km, fb, 64, it.g, z);
        tcx::tma_load_3d(dst + 2 * ATT_BOX, vm, fb, 0, it.g, z);
        tcx::tma_load_3d(dst + 3 * ATT_BOX, vm, fb, 64, it.g, z);
      }
      __syncwarp();
      ++st.tile_pos;
      ++st.cur_t;
    }
    if (st.cur_t >= n_t) {
      if (prefetch) return;   // publish (after the barrier) before claiming more
      st.cur = -1;
    }
  }
}

// attention consumers (warps 1-4, one 128-thread group, named barrier 2)
template <int G>
__device__ void att_consume(const Params& p, uint8_t* aring, AttShared& as, int64_t& tile_pos, int& ordinal,
                            int& merge_pos, const float* qq, float* sO, float* sML) {
  const int wg = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int tid = threadIdx.x - 32;   // 0..127
  const int gq = lane >> 2, tq = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  while (true) {
    const int q = ordinal % ITEMQ;
    bwait(p, smem_u32(&as.it_full[q]), uint32_t(ordinal / ITEMQ) & 1u, 1u << 6);
    const int item = as.item[q];
    ++ordinal;
    if (item < 0 || failed(p)) {
      named_sync(2, 128);
      if (tid == 0) tcx::mbar_arrive(smem_u32(&as.it_empty[q]));
      break;
    }
    const AttItem it = att_item(p, as, item);
    const int h0 = it.g * G;
    const float* qs = qq + q * G * HD;   // written by the producer before it published the item
    uint32_t qa[8][2];   // q fragments (rows = heads; rows >= G are zero)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 16 * kk + 2 * tq;
      qa[kk][0] = gq < G ? pack_bf16(qs[gq * HD + d0], qs[gq * HD + d0 + 1]) : 0u;
      qa[kk][1] = gq < G ? pack_bf16(qs[gq * HD + d0 + 8], qs[gq * HD + d0 + 9]) : 0u;
    }
    const int n_t = it.start < it.end ? (it.end - it.start + ATT_KT - 1) / ATT_KT : 0;
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;
    const int key0 = wg * 16;
    for (int t = 0; t < n_t; ++t, ++tile_pos) {
      const int stg = int(tile_pos % ATT_STAGES);
      const bool ok = bwait(p, smem_u32(&as.full[stg]), uint32_t(tile_pos / ATT_STAGES) & 1u, 1u << 7);
      uint8_t* tk = aring + size_t(stg) * ATT_STAGE;
      uint8_t* tv = tk + 2 * ATT_BOX;
      const int kbase = it.start + t * ATT_KT + key0;   // key position of this warp's first row
      if (kbase + 16 > it.end) {
        // keys past the item: zero their V rows (whatever the cache holds there)
        for (int i = 0; i < 16; ++i)
          if (kbase + i >= it.end && lane < 16)
            *reinterpret_cast<uint4*>(tv + kv_off(key0 + i, lane)) = make_uint4(0u, 0u, 0u, 0u);
        tcx::fence_proxy_async();
        __syncwarp();
      }
      float sc[2][4], sc2[2][4];   // two chains per n-tile (even / odd k steps)
#pragma unroll
      for (int n = 0; n < 2; ++n)
        sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = sc2[n][0] = sc2[n][1] = sc2[n][2] = sc2[n][3] = 0.0f;
      if (ok) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_u32(tk + kv_off(key0 + ri + 8 * (mi >> 1), 2 * kk + (mi & 1))), b0, b1, b2, b3);
          if (kk & 1) {
            mma16816(sc2[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
            mma16816(sc2[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
          } else {
            mma16816(sc[0], qa[kk][0], 0u, qa[kk][1], 0u, b0, b1);
            mma16816(sc[1], qa[kk][0], 0u, qa[kk][1], 0u, b2, b3);
          }
        }
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[n][e] += sc2[n][e];
      }
      float x[4];
      float mx = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int kp = kbase + 8 * n + 2 * tq + e;
          const float v = kp < it.end ? sc[n][e] * p.scale_log2 : -INFINITY;
          x[2 * n + e] = v;
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
      // P split into bf16 hi (A rows 0-7, the heads) and lo = bf16(p - hi)
      // (A rows 8-15, otherwise unused): accumulator rows 8-15 collect lo*V
      uint32_t a0, a1, a2, a3;
      split_p(pr, a0, a1, a2, a3);
      if (ok) {
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(tv + kv_off(key0 + ri + 8 * (mi & 1), 2 * dp + (mi >> 1))), b0, b1, b2, b3);
          mma16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
          mma16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) tcx::mbar_arrive(smem_u32(&as.empty[stg]));
    }
    // merge the four warps' softmax states of every head (dedicated scratch:
    // the ring may already hold the next item's tiles)
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (gq < G) {
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {   // the hi and lo parts of P * V
        sO[(wg * G + gq) * HD + 8 * dn + 2 * tq] = o[dn][0] + o[dn][2];
        sO[(wg * G + gq) * HD + 8 * dn + 2 * tq + 1] = o[dn][1] + o[dn][3];
      }
      if (tq == 0) {
        sML[(wg * G + gq) * 2] = m_run;
        sML[(wg * G + gq) * 2 + 1] = l_run;
      }
    }
    named_sync(2, 128);
    const int d = tid;
    const int bg = it.b * p.nkv + it.g;
    for (int j = 0; j < G; ++j) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, sML[(w * G + j) * 2]);
      float Ls = 0.0f, O = 0.0f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float mw = sML[(w * G + j) * 2];
          if (mw == -INFINITY) continue;
          const float sc = exp2f(mw - M);
          Ls += sML[(w * G + j) * 2 + 1] * sc;
          O += sO[(w * G + j) * HD + d] * sc;
        }
      }
      const int64_t idx = (int64_t(it.b) * p.nh + h0 + j) * p.att_splits + it.split;
      p.att_o[idx * HD + d] = O;
      if (d == 0) {
        p.att_ml[2 * idx] = M;
        p.att_ml[2 * idx + 1] = Ls;
      }
    }
    // hand the finished chunk to the merge warp (it counts chunks and merges the last)
    named_sync(2, 128);
    if (tid == 0) {
      const int mq = merge_pos % MERGEQ;
      if (merge_pos >= MERGEQ) bwait(p, smem_u32(&as.mq_empty[mq]), uint32_t(merge_pos / MERGEQ - 1) & 1u, 1u << 8);
      as.merge[mq] = bg;
      tcx::mbar_arrive(smem_u32(&as.mq_full[mq]));
      tcx::mbar_arrive(smem_u32(&as.it_empty[q]));
    }
    ++merge_pos;
  }
  // end of the stage for the merge warp
  if (tid == 0) {
    const int mq = merge_pos % MERGEQ;
    if (merge_pos >= MERGEQ) bwait(p, smem_u32(&as.mq_empty[mq]), uint32_t(merge_pos / MERGEQ - 1) & 1u, 1u << 8);
    as.merge[mq] = -1;
    tcx::mbar_arrive(smem_u32(&as.mq_full[mq]));
  }
  ++merge_pos;
}

// merge warp (warp 6): for each finished chunk, count it; the last chunk of
// a (sequence, kv head) merges every chunk of its G heads in chunk order.
template <int G>
__device__ void att_merge(const Params& p, AttShared& as, int& merge_pos) {
  const int lane = threadIdx.x & 31;
  while (true) {
    const int mq = merge_pos % MERGEQ;
    bwait(p, smem_u32(&as.mq_full[mq]), uint32_t(merge_pos / MERGEQ) & 1u, 1u << 9);
    const int bg = as.merge[mq];
    ++merge_pos;
    __syncwarp();
    if (lane == 0) tcx::mbar_arrive(smem_u32(&as.mq_empty[mq]));
    if (bg < 0 || failed(p)) break;
    unsigned int old = 0;
    if (lane == 0) {
      __threadfence();   // the consumer group's partials (ordered before the queue entry)
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p.cnt_att + bg) : "memory");
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old != unsigned(p.att_splits - 1)) continue;
    __threadfence();
    const int b = bg / p.nkv, g = bg % p.nkv;
    for (int j = 0; j < G; ++j) {
      const int64_t base = (int64_t(b) * p.nh + g * G + j) * p.att_splits;
      const bool in = lane < p.att_splits;   // lane s holds chunk s (splits <= 32)
      const float ms = in ? __ldcg(p.att_ml + 2 * (base + lane)) : -INFINITY;
      const float ls = in ? __ldcg(p.att_ml + 2 * (base + lane) + 1) : 0.0f;
      const float M = warp_max(ms);
      const float w = (ms == -INFINITY || M == -INFINITY) ? 0.0f : exp2f(ms - M);
      const float inv_l = 1.0f / fmaxf(warp_sum(ls * w), 1e-30f);
      float O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int sp = 0; sp < p.att_splits; ++sp) {
        const float ws = __shfl_sync(0xffffffffu, w, sp);
#pragma unroll
        for (int i = 0; i < 4; ++i) O[i] += __ldcg(p.att_o + (base + sp) * HD + lane + 32 * i) * ws;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        p.attn_buf[(int64_t(b) * p.nh + g * G + j) * HD + lane + 32 * i] = __float2bfloat16_rn(O[i] * inv_l);
    }
    if (lane == 0) p.cnt_att[bg] = 0u;
  }
}

template <int G>
__global__ void __launch_bounds__(THREADS, 1) decode_step_kernel(const __grid_constant__ Params p) {
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  // layout: union (attention ring | normed y | staged o_proj/down inputs) | weight ring |
  //         o_proj/down partials | q | merge scratch | barriers
  uint8_t* uni = sm;
  bf16* ys = reinterpret_cast<bf16*>(uni);
  uint8_t* wring = uni + p.union_bytes;
  float* red = reinterpret_cast<float*>(wring + size_t(p.ring) * SLOT);
  float* qq = red + size_t(p.red_units) * 16 * p.B;   // [ITEMQ][G][HD]
  float* sO = qq + ITEMQ * G * HD;
  float* sML = sO + 4 * G * HD;
  uint64_t* wfull = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(sML + 4 * G * 2) + 7) & ~uintptr_t(7));
  uint64_t* wempty = wfull + p.ring;
  AttShared& as = *reinterpret_cast<AttShared*>(wempty + p.ring);
  const int warp = threadIdx.x >> 5;
  unsigned long long bar_target = 0;   // grid barrier base: see grid_sync
  if (threadIdx.x == 32) bar_target = ld_acquire_u64(p.bar) / gridDim.x * gridDim.x;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.ring; ++i) {
      tcx::mbar_init(smem_u32(wfull + i), 1);
      tcx::mbar_init(smem_u32(wempty + i), 1);
    }
    for (int i = 0; i < ATT_STAGES; ++i) {
      tcx::mbar_init(smem_u32(&as.full[i]), 1);
      tcx::mbar_init(smem_u32(&as.empty[i]), 4);
    }
    for (int i = 0; i < ITEMQ; ++i) {
      tcx::mbar_init(smem_u32(&as.it_full[i]), 1);
      tcx::mbar_init(smem_u32(&as.it_empty[i]), 1);
    }
    for (int i = 0; i < MERGEQ; ++i) {
      tcx::mbar_init(smem_u32(&as.mq_full[i]), 1);
      tcx::mbar_init(smem_u32(&as.mq_empty[i]), 1);
    }
    tcx::fence_mbar_init();
    for (int l = 0; l < p.n_layers; ++l) {
      tcx::prefetch_map(&p.kmap[l]);
      tcx::prefetch_map(&p.vmap[l]);
    }
  }
  if (threadIdx.x >= 32 && threadIdx.x < 32 + p.B) {   // this step's per-token inputs
    const int b = threadIdx.x - 32;
    as.pos[b] = p.positions[b];
    as.slot[b] = p.slots[b];
    as.ctx[b] = p.ctx_lens[b];
    as.base[b] = p.seq_base[b];
  }
  __syncthreads();
  if (warp == 0) {
    producer(p, wring, wfull, wempty);
    return;
  }
  const int cw = warp - 1, lane = threadIdx.x & 31;
  int64_t pos = 0;                      // weight stream position of the next unit of this CTA
  AttProducer ap{0, 0, -1, 0, false, false};   // warp 5's state
  int64_t tile_pos = 0;                 // consumers' attention ring position
  int ordinal = 0;                     // consumers' item queue position
  int merge_pos = 0;                   // merge queue position (consumers and the merge warp)
  for (int l = 0; l < p.n_layers; ++l) {
    const int c0 = 2 * l, c1 = 2 * l + 1;   // residual updates of this layer
    norm_stage(p, l == 0 ? p.x : p.h_buf, l == 0 ? nullptr : p.res_buf + size_t((c0 - 1) & 1) * p.B * p.H,
               p.res_buf + size_t(c0 & 1) * p.B * p.H, p.layers[l].input_ln, ys);
    gemv_stage(p, G_QKV, pos, wring, wfull, wempty, ys, nullptr, nullptr, red);
    pos += gemv_of(p, G_QKV).units;
    ap.cur = -1;   // the item queue's and the ring's positions continue across layers (barrier phases do)
    ap.done = false;
    // every warp is done with ys (the ring may be refilled): arrive, let the
    // attention producer load cached history, then wait for everyone's QKV
    grid_arrive(p, bar_target);
    if (cw == 4) att_produce<G>(p, l, uni, as, qq, ap, true);
    grid_wait(p, bar_target);
    if (cw == 4) att_produce<G>(p, l, uni, as, qq, ap, false);
    else if (cw < 4) att_consume<G>(p, uni, as, tile_pos, ordinal, merge_pos, qq, sO, sML);
    else if (cw == 5) att_merge<G>(p, as, merge_pos);
    grid_sync(p, bar_target);
    gemv_stage(p, G_O, pos, wring, wfull, wempty, nullptr, p.attn_buf, reinterpret_cast<bf16*>(uni), red);
    pos += gemv_of(p, G_O).units;
    grid_sync(p, bar_target);
    norm_stage(p, p.h_buf, p.res_buf + size_t(c0 & 1) * p.B * p.H, p.res_buf + size_t(c1 & 1) * p.B * p.H,
               p.layers[l].post_ln, ys);
    gemv_stage(p, G_GU, pos, wring, wfull, wempty, ys, nullptr, nullptr, red);
    pos += gemv_of(p, G_GU).units;
    grid_sync(p, bar_target);
    gemv_stage(p, G_DOWN, pos, wring, wfull, wempty, nullptr, p.act_buf, reinterpret_cast<bf16*>(uni), red);
    pos += gemv_of(p, G_DOWN).units;
    grid_sync(p, bar_target);
  }
  // final RMSNorm of (h + residual): CTA b < B handles token b with one warp
  if (int(blockIdx.x) < p.B && cw == 0) {
    const int t = blockIdx.x;
    const bf16* res = p.res_buf + size_t((2 * p.n_layers - 1) & 1) * p.B * p.H;
    float ss = 0.0f;
    for (int k = lane * 8; k < p.H; k += 256) {
      const uint4 hv = ldcg16(p.h_buf + int64_t(t) * p.H + k);
      const uint4 rv = ldcg16(res + int64_t(t) * p.H + k);
      const bf16* hb = reinterpret_cast<const bf16*>(&hv);
      const bf16* rb = reinterpret_cast<const bf16*>(&rv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float v = round_t<bf16>(__bfloat162float(hb[e]) + __bfloat162float(rb[e]));
        ss += v * v;
      }
    }
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / float(p.H) + p.eps);
    for (int k = lane * 8; k < p.H; k += 256) {
      const uint4 hv = ldcg16(p.h_buf + int64_t(t) * p.H + k);
      const uint4 rv = ldcg16(res + int64_t(t) * p.H + k);
      const bf16* hb = reinterpret_cast<const bf16*>(&hv);
      const bf16* rb = reinterpret_cast<const bf16*>(&rv);
      float v[8], g[8];
      load16(p.final_ln + k, g);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        v[e] = (round_t<bf16>(__bfloat162float(hb[e]) + __bfloat162float(rb[e])) * inv) * g[e];
      store16(p.out + int64_t(t) * p.H + k, v);
    }
  }
  // every attention item of every layer has been claimed: reset the counters
  if (blockIdx.x == 0 && cw == 0)
    for (int l = lane; l < p.n_layers; l += 32) p.work[l] = 0u;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
struct Plan {
  int chunk, splits, ring, red_units;
  uint32_t union_bytes;
  size_t smem;
};
constexpr size_t kCountersBytes = 64 * 1024;
constexpr int kMaxSplits = 32;   // the split merge gives one lane to each chunk

// cap: dynamic shared memory a CTA may use (the opt-in limit minus the kernel's static shared memory)
Plan plan(int B, int H, int nh, int nkv, int I, int tp, int max_context, int sms, size_t cap) {
  Plan pl;
  const int G = nh / nkv;
  // attention items: about four per SM, chunks of whole tiles
  const int pairs = B * nkv;
  const int want = 4 * sms;
  const int splits = std::min(kMaxSplits, std::max(1, want / std::max(1, pairs)));
  int chunk = (max_context + splits - 1) / splits;
  chunk = std::max(ATT_KT, (chunk + ATT_KT - 1) / ATT_KT * ATT_KT);
  pl.chunk = chunk;
  pl.splits = (max_context + chunk - 1) / chunk;
  pl.red_units = 0;
  size_t xmax = size_t(B) * (H + YPAD) * 2;
  for (int w = 0; w < 4; ++w) {
    for (int c = 0; c < sms; ++c) {
      const Gemv g = gemv_geom(w, H, nh, nkv, I, tp, c, sms);
      if (w == G_O || w == G_DOWN) pl.red_units = std::max(pl.red_units, g.units);
    }
    const Gemv g = gemv_geom(w, H, nh, nkv, I, tp, 0, sms);
    if (w == G_O || w == G_DOWN) xmax = std::max(xmax, size_t(B) * (g.K + YPAD) * 2);
  }
  const size_t un = std::max(size_t(ATT_STAGES) * ATT_STAGE, xmax);
  pl.union_bytes = uint32_t((un + 1023) / 1024 * 1024);
  const size_t fixed = 1024 + pl.union_bytes + size_t(pl.red_units) * 16 * B * 4 + size_t(G) * HD * 4 * (ITEMQ + 4) +
                       size_t(G) * 8 * 4 + size_t(G) * 33 * 4 + 64 + sizeof(AttShared);
  pl.ring = cap > fixed ? int((cap - fixed) / (SLOT + 16)) : 0;
  pl.ring = std::min(pl.ring, 12);
  pl.smem = fixed + size_t(pl.ring) * (SLOT + 16);
  return pl;
}

struct WsLayout {
  size_t bar, err, work, cnt_att, att_o, att_ml, qkv, attn, act, h, res, total;
};
WsLayout ws_layout(int n_layers, int B, int H, int nh, int nkv, int I, int splits) {
  WsLayout w;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) / 256 * 256;
    return o;
  };
  const size_t qkvw = size_t(nh + 2 * nkv) * HD;
  w.bar = take(kCountersBytes);   // counters region: zero at allocation, left so by each call
  w.err = w.bar + 64;
  w.work = w.bar + 256;
  w.cnt_att = w.work + 4 * size_t(MAXL);
  w.att_o = take(size_t(B) * nh * splits * HD * 4);
  w.att_ml = take(size_t(B) * nh * splits * 2 * 4);
  w.qkv = take(size_t(B) * qkvw * 2);
  w.attn = take(size_t(B) * nh * HD * 2);
  w.act = take(size_t(B) * I * 2);
  w.h = take(size_t(B) * H * 2);
  w.res = take(size_t(2) * B * H * 2);
  w.total = off;
  (void)n_layers;
  return w;
}

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  });
  return n;
}

bool shape_ok(int B, int H, int nh, int nkv, int hd, int I, int tp) {
  if (B < 1 || B > MAXB || hd != HD || nh <= 0 || nkv <= 0 || tp <= 0 || I <= 0) return false;
  if (nh % nkv || nh % tp || nkv % tp || I % tp) return false;
  const int G = nh / nkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  // whole rows per shard in 16-byte pieces; every staged row fits one ring slot
  if (H % 256 || (nh * HD / tp) % 256 || (I / tp) % 256) return false;
  for (int w = 0; w < 4; ++w)
    if (gemv_geom(w, H, nh, nkv, I, tp, 0, 1).R < 1) return false;
  return true;
}

// dynamic shared memory available to decode_step_kernel<G>
template <int G>
size_t smem_cap() {
  static size_t cap = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes a{};
    if (cudaFuncGetAttributes(&a, decode_step_kernel<G>) == cudaSuccess && size_t(optin) > a.sharedSizeBytes + 128)
      cap = size_t(optin) - a.sharedSizeBytes - 128;
  });
  return cap;
}
size_t smem_cap_for(int G) {
  switch (G) {
    case 1: return smem_cap<1>();
    case 2: return smem_cap<2>();
    case 4: return smem_cap<4>();
    default: return smem_cap<8>();
  }
}

template <int G>
int launch(const Params& p, size_t smem, cudaStream_t st) {
  // the shared memory a launch needs depends on B: allow the ceiling once
  static bool configured = false;
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_step_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem_cap<G>()));
    if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  if (smem > smem_cap<G>()) return set_error(QW_ERR_SHAPE, "qw_decode_layers: needs %zu bytes of shared memory", smem);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(sm_count()));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_step_kernel<G>, p);
  if (e != cudaSuccess) return set_error(QW_ERR_CUDA, "decode_step_kernel launch: %s", cudaGetErrorString(e));
  return QW_OK;
}

}  // namespace dstep

unsigned int take_dstep_errors() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, dstep::g_dstep_error, sizeof(v));
  if (v) cudaMemcpyToSymbol(dstep::g_dstep_error, &z, sizeof(z));
  return v;
}

}  // namespace qw

using namespace qw;

static_assert(sizeof(qw_decode_layer) == sizeof(dstep::LayerPtrs), "qw_decode_layer layout");

extern "C" size_t qw_decode_layers_workspace_size(int n_layers, int B, int H, int n_heads, int n_kv_heads,
                                                  int head_dim, int intermediate, int tp, int max_context) {
  if (n_layers <= 0 || n_layers > dstep::MAXL || max_context <= 0 ||
      !dstep::shape_ok(B, H, n_heads, n_kv_heads, head_dim, intermediate, tp))
    return 0;
  const int sms = dstep::sm_count() > 0 ? dstep::sm_count() : 1;
  const dstep::Plan pl = dstep::plan(B, H, n_heads, n_kv_heads, intermediate, tp, max_context, sms, 0);
  return dstep::ws_layout(n_layers, B, H, n_heads, n_kv_heads, intermediate, pl.splits).total;
}

extern "C" int qw_decode_layers(const qw_decode_layer* layers, int n_layers, const void* x, const int64_t* positions,
                                const int64_t* slot_mapping, const int32_t* context_lens, const int32_t* seq_base,
                                int B, int max_context, int H, int n_heads, int n_kv_heads, int head_dim,
                                int intermediate, int tp, const float* cos_sin, int64_t max_position,
                                int64_t num_slots, float eps, float scale, const void* final_norm, void* out,
                                int32_t* err_count, void* workspace, size_t workspace_bytes, void* stream) {
  if (n_layers <= 0 || n_layers > dstep::MAXL || max_context <= 0 || num_slots <= 0)
    return set_error(QW_ERR_INVALID_ARG, "qw_decode_layers: bad n_layers, max_context or num_slots");
  if (!dstep::shape_ok(B, H, n_heads, n_kv_heads, head_dim, intermediate, tp))
    return set_error(QW_ERR_SHAPE, "qw_decode_layers: unsupported shape (B %d, H %d, nh %d, nkv %d, hd %d, I %d, tp %d)",
                     B, H, n_heads, n_kv_heads, head_dim, intermediate, tp);
  if (!layers || !x || !positions || !slot_mapping || !context_lens || !seq_base || !cos_sin || !final_norm || !out ||
      !workspace)
    return set_error(QW_ERR_INVALID_ARG, "qw_decode_layers: null pointer");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(workspace) |
       reinterpret_cast<uintptr_t>(final_norm)) % 16)
    return set_error(QW_ERR_INVALID_ARG, "qw_decode_layers: x, out, final_norm and workspace must be 16-byte aligned");
  for (int l = 0; l < n_layers; ++l) {
    const qw_decode_layer& lw = layers[l];
    if (!lw.input_layernorm || !lw.qkv || !lw.q_norm || !lw.k_norm || !lw.o_proj || !lw.post_attention_layernorm ||
        !lw.gate_up || !lw.down || !lw.k_cache || !lw.v_cache)
      return set_error(QW_ERR_INVALID_ARG, "qw_decode_layers: layer %d has a null pointer", l);
    if ((reinterpret_cast<uintptr_t>(lw.qkv) | reinterpret_cast<uintptr_t>(lw.o_proj) |
         reinterpret_cast<uintptr_t>(lw.gate_up) | reinterpret_cast<uintptr_t>(lw.down) |
         reinterpret_cast<uintptr_t>(lw.k_cache) | reinterpret_cast<uintptr_t>(lw.v_cache)) % 16)
      return set_error(QW_ERR_INVALID_ARG, "qw_decode_layers: layer %d weights and caches must be 16-byte aligned", l);
  }
  const int G = n_heads / n_kv_heads;
  const int sms = dstep::sm_count();
  if (sms <= 0) return set_error(QW_ERR_CUDA, "qw_decode_layers: no device");
  const dstep::Plan pl =
      dstep::plan(B, H, n_heads, n_kv_heads, intermediate, tp, max_context, sms, dstep::smem_cap_for(G));
  if (pl.ring < 2) return set_error(QW_ERR_SHAPE, "qw_decode_layers: shared memory too small for this shape");
  const dstep::WsLayout wl = dstep::ws_layout(n_layers, B, H, n_heads, n_kv_heads, intermediate, pl.splits);
  if (workspace_bytes < wl.total)
    return set_error(QW_ERR_WORKSPACE, "qw_decode_layers: workspace %zu < %zu bytes", workspace_bytes, wl.total);
  // the kernel parameters (passed by value: a CUDA graph keeps its own copy)
  static dstep::Params p;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(static_cast<void*>(&p), 0, sizeof(p));
  for (int l = 0; l < n_layers; ++l) {
    std::memcpy(static_cast<void*>(&p.layers[l]), &layers[l], sizeof(dstep::LayerPtrs));
    const uint64_t dims[3] = {uint64_t(head_dim), uint64_t(n_kv_heads), uint64_t(num_slots)};
    const uint64_t strides[2] = {uint64_t(head_dim) * 2, uint64_t(n_kv_heads) * head_dim * 2};
    const uint32_t box[3] = {64u, 1u, uint32_t(dstep::ATT_KT)};
    int rc = make_tensor_map(&p.kmap[l], layers[l].k_cache, 3, dims, strides, box);
    if (rc) return rc;
    rc = make_tensor_map(&p.vmap[l], layers[l].v_cache, 3, dims, strides, box);
    if (rc) return rc;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.n_layers = n_layers;
  p.B = B;
  p.H = H;
  p.nh = n_heads;
  p.nkv = n_kv_heads;
  p.I = intermediate;
  p.tp = tp;
  p.x = static_cast<const bf16*>(x);
  p.final_ln = static_cast<const bf16*>(final_norm);
  p.out = static_cast<bf16*>(out);
  p.positions = positions;
  p.slots = slot_mapping;
  p.ctx_lens = context_lens;
  p.seq_base = seq_base;
  p.cos_sin = cos_sin;
  p.max_pos = max_position;
  p.num_slots = num_slots;
  p.eps = eps;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.att_chunk = pl.chunk;
  p.att_splits = pl.splits;
  p.ring = pl.ring;
  p.red_units = pl.red_units;
  p.union_bytes = pl.union_bytes;
  p.bar = reinterpret_cast<unsigned long long*>(ws + wl.bar);
  p.err = reinterpret_cast<unsigned int*>(ws + wl.err);
  p.work = reinterpret_cast<unsigned int*>(ws + wl.work);
  p.cnt_att = reinterpret_cast<unsigned int*>(ws + wl.cnt_att);
  p.err_count = err_count;
  p.att_o = reinterpret_cast<float*>(ws + wl.att_o);
  p.att_ml = reinterpret_cast<float*>(ws + wl.att_ml);
  p.qkv_buf = reinterpret_cast<bf16*>(ws + wl.qkv);
  p.attn_buf = reinterpret_cast<bf16*>(ws + wl.attn);
  p.act_buf = reinterpret_cast<bf16*>(ws + wl.act);
  p.h_buf = reinterpret_cast<bf16*>(ws + wl.h);
  p.res_buf = reinterpret_cast<bf16*>(ws + wl.res);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (G) {
    case 1: return dstep::launch<1>(p, pl.smem, st);
    case 2: return dstep::launch<2>(p, pl.smem, st);
    case 4: return dstep::launch<4>(p, pl.smem, st);
    default: return dstep::launch<8>(p, pl.smem, st);
  }
}
