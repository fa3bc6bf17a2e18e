// CUDA-core kernels: backward preprocess, dQ convert, the fp32 backward, the
// forward, and the keep-mask generator.
//
// The arithmetic follows the formulas section of the FAG-V2 page
// (aclnnFlashAttentionUnpaddingScoreGradV2, 功能说明 / 计算公式):
// S = scale Q K^T (masked), P = softmax(S) with dropout, Y = P V, dV = P^T dY,
// dQ = scale dS K, dK = scale dS^T Q, dS = P (dP Z / keep_prob - D).

#include <cuda_runtime.h>
#include <math_constants.h>

#include "common.cuh"

namespace fav {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// preprocess: D_i = sum_d dY * Y, lse2_i = (max_i + ln sum_i) * log2(e)
// (the tensor-core kernel with dropout takes D_i * keep_prob and
// lse2_i + log2(keep_prob): BwdParams::dsum_scale, lse2_shift),
// dq_acc row := 0, the tile's deterministic-mode dQ counter := 0.  One block
// per (64-row padded query tile, head).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void clear_dq_counter(const BwdParams &p, int tile, int n) {
  if (threadIdx.x == 0) p.sem[int64_t(n) * (p.tp / kQTile) + tile] = 0;
}

template <typename T>
__device__ __forceinline__ float dot16(uint4 a, uint4 b) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
  if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int k = 0; k < 4; ++k) acc = fmaf(__uint_as_float(av[k]), __uint_as_float(bv[k]), acc);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const T *ah = reinterpret_cast<const T *>(&av[k]);
      const T *bh = reinterpret_cast<const T *>(&bv[k]);
      acc = fmaf(to_f(ah[0]), to_f(bh[0]), acc);
      acc = fmaf(to_f(ah[1]), to_f(bh[1]), acc);
    }
  }
  return acc;
}

// Rows are read with 16-byte loads, D / (16 / sizeof(T)) lanes per row and
// several rows per warp instruction.  The block first issues its dq_acc
// zero stores, then every load of its rows (dY, Y and the statistics)
// before any reduction, so that all its memory traffic is in flight at
// once.  Needs 16-byte aligned dY and Y (the launcher checks; otherwise
// preprocess_kernel below runs).
template <typename T, int D>
__global__ void __launch_bounds__(256) preprocess_vec_kernel(BwdParams p) {
  constexpr int kVec = 16 / int(sizeof(T));
  constexpr int kLanes = D / kVec;
  constexpr int kRowsPass = 32 / kLanes;
  constexpr int kRowsWarp = kQTile / 8;
  constexpr int kPasses = kRowsWarp / kRowsPass;
  const int tile = blockIdx.x, n = blockIdx.y;
  const int row0 = tile * kQTile;
  const int b = seq_of_padded_row(p.seqs, p.batch, row0);
  const SeqInfo s = p.seqs[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / kLanes, part = lane % kLanes;
  const uint4 *dy = static_cast<const uint4 *>(p.dy);
  const uint4 *y = static_cast<const uint4 *>(p.y);
  clear_dq_counter(p, tile, n);
  for (int e = threadIdx.x; e < kQTile * (D / 4); e += 256) {
    const int r = e / (D / 4), c4 = e % (D / 4);
    const int i = row0 + r - s.qpad;
    if (i < s.len_q)
      reinterpret_cast<float4 *>(p.dq_acc + ((int64_t(s.cu_q) + i) * p.n + n) * D)[c4] =
          make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint4 a[kPasses], c[kPasses];
  float mm[kPasses], ll[kPasses];
#pragma unroll
  for (int k = 0; k < kPasses; ++k) {
    const int i = row0 + warp * kRowsWarp + k * kRowsPass + sub - s.qpad;
    a[k] = c[k] = make_uint4(0u, 0u, 0u, 0u);
    mm[k] = -CUDART_INF_F; ll[k] = 0.f;
    if (i < s.len_q) {
      const int64_t t = int64_t(s.cu_q) + i;
      const int64_t e = (t * p.n + n) * (D / kVec) + part;
      a[k] = __ldg(dy + e);
      c[k] = __ldg(y + e);
      if (part == 0) {
        mm[k] = __ldg(p.smax + (t * p.n + n) * 8);
        ll[k] = __ldg(p.ssum + (t * p.n + n) * 8);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < kPasses; ++k) {
    const int prow = row0 + warp * kRowsWarp + k * kRowsPass + sub;
    const int i = prow - s.qpad;
    float acc = dot16<T>(a[k], c[k]);
#pragma unroll
    for (int o = kLanes / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (part == 0) {
      float lse2 = CUDART_INF_F;
      if (i < s.len_q) {
        const float m = mm[k], l = ll[k];
        if (l > 0.f && m > -CUDART_INF_F) lse2 = (m + logf(l)) * kLog2e + p.lse2_shift;
        acc *= p.dsum_scale;
      } else {
        acc = 0.f;
      }
      p.lse2[int64_t(n) * p.tp + prow] = lse2;
      p.dsum[int64_t(n) * p.tp + prow] = acc;
    }
  }
}

// Same results for any alignment: one warp per row.
template <typename T, int D>
__global__ void __launch_bounds__(256) preprocess_kernel(BwdParams p) {
  const int tile = blockIdx.x, n = blockIdx.y;
  const int row0 = tile * kQTile;
  const int b = seq_of_padded_row(p.seqs, p.batch, row0);
  const SeqInfo s = p.seqs[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T *dy = static_cast<const T *>(p.dy);
  const T *y = static_cast<const T *>(p.y);
  clear_dq_counter(p, tile, n);
  for (int r = warp; r < kQTile; r += 8) {
    const int prow = row0 + r;
    const int i = prow - s.qpad;
    float dsum = 0.f, lse2 = CUDART_INF_F;
    if (i < s.len_q) {
      const int64_t t = int64_t(s.cu_q) + i;
      const int64_t base = (t * p.n + n) * D;
      float acc = 0.f;
#pragma unroll
      for (int d = lane; d < D; d += 32) acc += to_f(dy[base + d]) * to_f(y[base + d]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      dsum = acc * p.dsum_scale;
      const float m = p.smax[(t * p.n + n) * 8];
      const float l = p.ssum[(t * p.n + n) * 8];
      if (l > 0.f && m > -CUDART_INF_F) lse2 = (m + logf(l)) * kLog2e + p.lse2_shift;
      float4 *acc_row = reinterpret_cast<float4 *>(p.dq_acc + base);
      for (int d4 = lane; d4 < D / 4; d4 += 32) acc_row[d4] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (lane == 0) {
      p.lse2[int64_t(n) * p.tp + prow] = lse2;
      p.dsum[int64_t(n) * p.tp + prow] = dsum;
    }
  }
}

// dQ = scale * dq_acc, cast to the storage type.
template <typename T>
__global__ void dq_convert_kernel(const float *__restrict__ acc, T *__restrict__ dq, int64_t n4,
                                  float scale) {
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n4;
       e += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4 *>(acc)[e];
    T *o = dq + e * 4;
    o[0] = from_f<T>(a.x * scale);
    o[1] = from_f<T>(a.y * scale);
    o[2] = from_f<T>(a.z * scale);
    o[3] = from_f<T>(a.w * scale);
  }
}

// Same, eight elements per thread with one 16-byte store (dq 16-byte aligned).
template <typename T>
__global__ void dq_convert8_kernel(const float *__restrict__ acc, T *__restrict__ dq, int64_t n8,
                                   float scale) {
  for (int64_t e = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; e < n8;
       e += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(acc) + 2 * e);
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(acc) + 2 * e + 1);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if constexpr (sizeof(T) == 4) {
      float4 *o = reinterpret_cast<float4 *>(dq) + 2 * e;
      o[0] = make_float4(v[0] * scale, v[1] * scale, v[2] * scale, v[3] * scale);
      o[1] = make_float4(v[4] * scale, v[5] * scale, v[6] * scale, v[7] * scale);
    } else {
      T h[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) h[i] = from_f<T>(v[i] * scale);
      uint4 u;
      memcpy(&u, h, sizeof(u));
      reinterpret_cast<uint4 *>(dq)[e] = u;
    }
  }
}

// ---------------------------------------------------------------------------
// Backward on CUDA cores.  One block per work item: 64 keys of one
// (sequence, key/value head), looping over the query heads of the group and
// the query tiles of 64 the window reaches.  dK, dV accumulate in registers;
// dQ partials go to dq_acc with fp32 atomics.
// Thread (ty, tx) of a 16 x 16 grid owns rows ty + 16a and columns tx + 16b.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_simt_kernel(BwdParams p) {
  constexpr int LD = D + 1;
  constexpr int PD = kQTile + 1;
  constexpr int DC = D / 16;
  extern __shared__ float smem[];
  float *Ks = smem;
  float *Vs = Ks + 64 * LD;
  float *Qs = Vs + 64 * LD;
  float *dYs = Qs + 64 * LD;
  float *Ps = dYs + 64 * LD;     // Pd[i][j]
  float *dSs = Ps + 64 * PD;     // dS[i][j]
  float *lse_s = dSs + 64 * PD;
  float *dsum_s = lse_s + 64;

  __shared__ int s_item, s_ok;
  if (threadIdx.x == 0) s_item = take_item(p);
  __syncthreads();
  const WorkItem it = p.items[s_item];
  const SeqInfo s = p.seqs[it.seq];
  const int kvh = it.head;
  const int group = p.n / p.n_kv;
  const int k0 = it.tile * kSimtKvTile;
  const int qlo = item_lo(it), qcnt = item_count(it);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const T *Q = static_cast<const T *>(p.q);
  const T *K = static_cast<const T *>(p.k);
  const T *V = static_cast<const T *>(p.v);
  const T *dY = static_cast<const T *>(p.dy);

  for (int e = tid; e < 64 * D; e += 256) {
    const int r = e / D, c = e % D;
    float kv = 0.f, vv = 0.f;
    if (k0 + r < s.len_k) {
      const int64_t off = ((int64_t(s.cu_k) + k0 + r) * p.n_kv + kvh) * D + c;
      kv = to_f(K[off]);
      vv = to_f(V[off]);
    }
    Ks[r * LD + c] = kv;
    Vs[r * LD + c] = vv;
  }

  float accK[4][DC], accV[4][DC];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < DC; ++c) accK[a][c] = accV[a][c] = 0.f;

  for (int h = 0; h < group; ++h) {
    const int n = kvh * group + h;
    for (int qt = qlo; qt < qlo + qcnt; ++qt) {
      const int q0 = qt * kQTile;
      __syncthreads();
      for (int e = tid; e < 64 * D; e += 256) {
        const int r = e / D, c = e % D;
        float qv = 0.f, dv = 0.f;
        if (q0 + r < s.len_q) {
          const int64_t off = ((int64_t(s.cu_q) + q0 + r) * p.n + n) * D + c;
          qv = to_f(Q[off]);
          dv = to_f(dY[off]);
        }
        Qs[r * LD + c] = qv;
        dYs[r * LD + c] = dv;
      }
      if (tid < 64) {
        lse_s[tid] = p.lse2[int64_t(n) * p.tp + s.qpad + q0 + tid];
        dsum_s[tid] = p.dsum[int64_t(n) * p.tp + s.qpad + q0 + tid];
      }
      __syncthreads();

      // S = Q K^T and dP = dY V^T for i = ty + 16a, j = tx + 16b.
      float sa[4][4], pa[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) sa[a][b] = pa[a][b] = 0.f;
#pragma unroll 4
      for (int d = 0; d < D; ++d) {
        float qv[4], gv[4], kv[4], vv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          qv[a] = Qs[(ty + 16 * a) * LD + d];
          gv[a] = dYs[(ty + 16 * a) * LD + d];
          kv[a] = Ks[(tx + 16 * a) * LD + d];
          vv[a] = Vs[(tx + 16 * a) * LD + d];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            sa[a][b] = fmaf(qv[a], kv[b], sa[a][b]);
            pa[a][b] = fmaf(gv[a], vv[b], pa[a][b]);
          }
      }
      // P from the saved statistics, dropout, dS.
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = ty + 16 * a;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int j = tx + 16 * b;
          const int gi = q0 + i, gj = k0 + j;
          float pv = 0.f, zs = 1.f;
          if (window_ok(gi, gj, s.len_q, s.len_k, s.pre, s.next) &&
              !atten_masked(p.atten_mask, p.am_cols, gi, gj)) {
            pv = exp2f(sa[a][b] * p.scale_log2 - lse_s[i]);
            if (p.use_dropout)
              zs = keep_bit(p.mask, s.mask_off, n, s.len_q, s.len_k, gi, gj) * p.inv_keep;
          }
          Ps[i * PD + j] = pv * zs;
          dSs[i * PD + j] = pv * (pa[a][b] * zs - dsum_s[i]);
        }
      }
      __syncthreads();

      // dV += Pd^T dY, dK += dS^T Q for j = ty + 16a, d = tx + 16c.
#pragma unroll 2
      for (int i = 0; i < kQTile; ++i) {
        float pv[4], sv[4], gv[DC], qv[DC];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          pv[a] = Ps[i * PD + ty + 16 * a];
          sv[a] = dSs[i * PD + ty + 16 * a];
        }
#pragma unroll
        for (int c = 0; c < DC; ++c) {
          gv[c] = dYs[i * LD + tx + 16 * c];
          qv[c] = Qs[i * LD + tx + 16 * c];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < DC; ++c) {
            accV[a][c] = fmaf(pv[a], gv[c], accV[a][c]);
            accK[a][c] = fmaf(sv[a], qv[c], accK[a][c]);
          }
      }

      // dQ partial = dS K for i = ty + 16a, d = tx + 16c, added into dq_acc.
      float dq[4][DC];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < DC; ++c) dq[a][c] = 0.f;
#pragma unroll 2
      for (int j = 0; j < kSimtKvTile; ++j) {
        float sv[4], kv[DC];
#pragma unroll
        for (int a = 0; a < 4; ++a) sv[a] = dSs[(ty + 16 * a) * PD + j];
#pragma unroll
        for (int c = 0; c < DC; ++c) kv[c] = Ks[j * LD + tx + 16 * c];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int c = 0; c < DC; ++c) dq[a][c] = fmaf(sv[a], kv[c], dq[a][c]);
      }
      // Deterministic mode: add after the key tiles above this one (the
      // order is descending), then let the next one in.
      int32_t *ctr = nullptr;
      int rank = 0;
      if (p.deterministic) {
        ctr = dq_counter(p, s, n, qt);
        rank = dq_rank(p, s, it.tile, qt);
        if (tid == 0) s_ok = wait_counter(ctr, rank, p.timeout_ns, nullptr);
        __syncthreads();
        if (!s_ok) {
          if (tid == 0) atomicCAS(p.err, 0, kErrTimeoutBase + kRoleSimtDq);
          return;
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int gi = q0 + ty + 16 * a;
        if (gi < s.len_q) {
          float *row = p.dq_acc + ((int64_t(s.cu_q) + gi) * p.n + n) * D;
#pragma unroll
          for (int c = 0; c < DC; ++c) atomicAdd(row + tx + 16 * c, dq[a][c]);
        }
      }
      if (p.deterministic) {
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release_gpu(ctr, rank + 1);
      }
    }
  }

  T *dK = static_cast<T *>(p.dk);
  T *dV = static_cast<T *>(p.dv);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int j = ty + 16 * a;
    if (k0 + j < s.len_k) {
      const int64_t off = ((int64_t(s.cu_k) + k0 + j) * p.n_kv + kvh) * D;
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        dK[off + tx + 16 * c] = from_f<T>(accK[a][c] * p.scale);
        dV[off + tx + 16 * c] = from_f<T>(accV[a][c]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Forward on CUDA cores (online softmax).  One block per (sequence, query
// head, 64-query tile), looping over key tiles of 64.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(256) fwd_simt_kernel(FwdParams p) {
  constexpr int LD = D + 1;
  constexpr int PD = kSimtKvTile + 1;
  constexpr int DC = D / 16;
  extern __shared__ float smem[];
  float *Qs = smem;
  float *Ks = Qs + 64 * LD;
  float *Vs = Ks + 64 * LD;
  float *Ps = Vs + 64 * LD;

  const WorkItem it = p.items[blockIdx.x];
  const SeqInfo s = p.seqs[it.seq];
  const int n = it.head;
  const int kvh = n / (p.n / p.n_kv);
  const int q0 = it.tile * kQTile;
  const int klo = item_lo(it), kcnt = item_count(it);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const T *Q = static_cast<const T *>(p.q);
  const T *K = static_cast<const T *>(p.k);
  const T *V = static_cast<const T *>(p.v);

  for (int e = tid; e < 64 * D; e += 256) {
    const int r = e / D, c = e % D;
    Qs[r * LD + c] = (q0 + r < s.len_q)
                         ? to_f(Q[((int64_t(s.cu_q) + q0 + r) * p.n + n) * D + c]) : 0.f;
  }
  float m[4], l[4], o[4][DC];
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    m[a] = -CUDART_INF_F;
    l[a] = 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) o[a][c] = 0.f;
  }

  for (int kt = klo; kt < klo + kcnt; ++kt) {
    const int k0 = kt * kSimtKvTile;
    __syncthreads();
    for (int e = tid; e < 64 * D; e += 256) {
      const int r = e / D, c = e % D;
      float kv = 0.f, vv = 0.f;
      if (k0 + r < s.len_k) {
        const int64_t off = ((int64_t(s.cu_k) + k0 + r) * p.n_kv + kvh) * D + c;
        kv = to_f(K[off]);
        vv = to_f(V[off]);
      }
      Ks[r * LD + c] = kv;
      Vs[r * LD + c] = vv;
    }
    __syncthreads();
    float sa[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) sa[a][b] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      float qv[4], kv[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        qv[a] = Qs[(ty + 16 * a) * LD + d];
        kv[a] = Ks[(tx + 16 * a) * LD + d];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) sa[a][b] = fmaf(qv[a], kv[b], sa[a][b]);
    }
    // online softmax: rows ty + 16a are shared by the 16 lanes with this ty.
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int gi = q0 + ty + 16 * a;
      float sv[4], mx = -CUDART_INF_F;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int gj = k0 + tx + 16 * b;
        const bool ok = window_ok(gi, gj, s.len_q, s.len_k, s.pre, s.next) &&
                        !atten_masked(p.atten_mask, p.am_cols, gi, gj);
        sv[b] = ok ? sa[a][b] * p.scale : -CUDART_INF_F;
        mx = fmaxf(mx, sv[b]);
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[a], mx);
      const float msafe = mnew == -CUDART_INF_F ? 0.f : mnew;
      const float corr = exp2f((m[a] - msafe) * kLog2e);
      float rs = 0.f;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float pv = exp2f((sv[b] - msafe) * kLog2e);
        rs += pv;
        float zs = 1.f;
        if (p.use_dropout && pv > 0.f)
          zs = keep_bit(p.mask, s.mask_off, n, s.len_q, s.len_k, gi, k0 + tx + 16 * b) *
               p.inv_keep;
        Ps[(ty + 16 * a) * PD + tx + 16 * b] = pv * zs;
      }
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) rs += __shfl_xor_sync(0xffffffffu, rs, off);
      l[a] = l[a] * corr + rs;
      m[a] = mnew;
#pragma unroll
      for (int c = 0; c < DC; ++c) o[a][c] *= corr;
    }
    __syncthreads();
#pragma unroll 2
    for (int j = 0; j < kSimtKvTile; ++j) {
      float pv[4], vv[DC];
#pragma unroll
      for (int a = 0; a < 4; ++a) pv[a] = Ps[(ty + 16 * a) * PD + j];
#pragma unroll
      for (int c = 0; c < DC; ++c) vv[c] = Vs[j * LD + tx + 16 * c];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < DC; ++c) o[a][c] = fmaf(pv[a], vv[c], o[a][c]);
    }
  }

  T *Y = static_cast<T *>(p.y);
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int gi = q0 + ty + 16 * a;
    if (gi < s.len_q) {
      const int64_t t = int64_t(s.cu_q) + gi;
      const float inv = l[a] > 0.f ? 1.f / l[a] : 0.f;
#pragma unroll
      for (int c = 0; c < DC; ++c) Y[(t * p.n + n) * D + tx + 16 * c] = from_f<T>(o[a][c] * inv);
      if (tx < 8) {
        p.smax[(t * p.n + n) * 8 + tx] = l[a] > 0.f ? m[a] : -CUDART_INF_F;
        p.ssum[(t * p.n + n) * 8 + tx] = l[a];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// SplitMix64 keep bits (synthetic-input utility).  Thread e writes bytes
// [4e, 4e + 4) of the mask.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t index) {
  uint64_t z = seed + (index + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void gen_keep_mask_kernel(uint8_t *mask, int64_t nbits, uint64_t seed, uint64_t thr,
                                     int keep_all) {
  const int64_t nbytes = (nbits + 7) >> 3;
  const int64_t nwords = (nbytes + 3) >> 2;
  for (int64_t w = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; w < nwords;
       w += int64_t(gridDim.x) * blockDim.x) {
    uint32_t word = 0;
    for (int k = 0; k < 32; ++k) {
      const int64_t g = w * 32 + k;
      const bool keep = g < nbits && (keep_all || splitmix64(seed, uint64_t(g)) < thr);
      word |= uint32_t(keep) << k;
    }
    const int64_t b0 = w * 4;
    if (b0 + 4 <= nbytes && (reinterpret_cast<uintptr_t>(mask) & 3) == 0) {
      reinterpret_cast<uint32_t *>(mask)[w] = word;
    } else {
      for (int k = 0; k < 4 && b0 + k < nbytes; ++k) mask[b0 + k] = uint8_t(word >> (8 * k));
    }
  }
}

template <typename T, int D>
cudaError_t launch_bwd_simt_t(const BwdParams &p, cudaStream_t st) {
  constexpr int smem = (4 * 64 * (D + 1) + 2 * 64 * (kQTile + 1) + 128) * int(sizeof(float));
  static_assert(D % 16 == 0 && smem <= 227 * 1024, "CUDA-core backward tiles");
  cudaError_t e = cudaFuncSetAttribute(bwd_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  bwd_simt_kernel<T, D><<<p.n_items, 256, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_fwd_simt_t(const FwdParams &p, cudaStream_t st) {
  const int smem = (3 * 64 * (D + 1) + 64 * (kSimtKvTile + 1)) * int(sizeof(float));
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  fwd_simt_kernel<T, D><<<p.n_items, 256, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_pre_t(const BwdParams &p, cudaStream_t st) {
  dim3 grid(p.tp / kQTile, p.n);
  // The 16-byte-load kernel packs whole rows into a warp: it needs the lanes
  // of one row to divide 32.
  constexpr int kLanes = D / (16 / int(sizeof(T)));
  constexpr bool kVecShape = kLanes <= 32 && 32 % kLanes == 0 && (kQTile / 8) % (32 / kLanes) == 0;
  if constexpr (kVecShape) {
    if (((reinterpret_cast<uintptr_t>(p.dy) | reinterpret_cast<uintptr_t>(p.y)) & 15u) == 0) {
      preprocess_vec_kernel<T, D><<<grid, 256, 0, st>>>(p);
      return cudaGetLastError();
    }
  }
  preprocess_kernel<T, D><<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_conv_t(const BwdParams &p, cudaStream_t st) {
  const int64_t n = int64_t(p.total_q) * p.n * p.d;   // a multiple of 32 (D is)
  if ((reinterpret_cast<uintptr_t>(p.dq) & 15u) == 0) {
    int64_t blocks = (n / 8 + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    if (blocks < 1) blocks = 1;
    dq_convert8_kernel<T><<<int(blocks), 256, 0, st>>>(p.dq_acc, static_cast<T *>(p.dq), n / 8,
                                                       p.scale);
    return cudaGetLastError();
  }
  int64_t blocks = (n / 4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  dq_convert_kernel<T><<<int(blocks), 256, 0, st>>>(p.dq_acc, static_cast<T *>(p.dq), n / 4,
                                                    p.scale);
  return cudaGetLastError();
}

// Head dims built for the CUDA-core kernels (multiples of 16, up to the
// largest whose backward tiles fit in 227 KB of shared memory).
#define FAV_DISPATCH_D(dt, d, DV, FN, ...)                                                \
  if ((d) == DV) {                                                                        \
    if ((dt) == FA_DTYPE_FP32) return FN<float, DV>(__VA_ARGS__);                         \
    if ((dt) == FA_DTYPE_BF16) return FN<__nv_bfloat16, DV>(__VA_ARGS__);                 \
    if ((dt) == FA_DTYPE_FP16) return FN<__half, DV>(__VA_ARGS__);                        \
  }
#define FAV_DISPATCH(dt, d, FN, ...)                                                      \
  do {                                                                                    \
    FAV_DISPATCH_D(dt, d, 32, FN, __VA_ARGS__)                                            \
    FAV_DISPATCH_D(dt, d, 64, FN, __VA_ARGS__)                                            \
    FAV_DISPATCH_D(dt, d, 96, FN, __VA_ARGS__)                                            \
    FAV_DISPATCH_D(dt, d, 128, FN, __VA_ARGS__)                                           \
    FAV_DISPATCH_D(dt, d, 192, FN, __VA_ARGS__)                                           \
    return cudaErrorInvalidValue;                                                         \
  } while (0)

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdParams &p, fa_dtype dt, cudaStream_t s) {
  FAV_DISPATCH(dt, p.d, launch_pre_t, p, s);
}

cudaError_t launch_bwd_simt(const BwdParams &p, fa_dtype dt, cudaStream_t s) {
  FAV_DISPATCH(dt, p.d, launch_bwd_simt_t, p, s);
}

cudaError_t launch_fwd_simt(const FwdParams &p, fa_dtype dt, cudaStream_t s) {
  FAV_DISPATCH(dt, p.d, launch_fwd_simt_t, p, s);
}

cudaError_t launch_dq_convert(const BwdParams &p, fa_dtype dt, cudaStream_t s) {
  if (dt == FA_DTYPE_FP32) return launch_conv_t<float>(p, s);
  if (dt == FA_DTYPE_BF16) return launch_conv_t<__nv_bfloat16>(p, s);
  if (dt == FA_DTYPE_FP16) return launch_conv_t<__half>(p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gen_keep_mask(uint8_t *mask, int64_t nbits, uint64_t seed, uint64_t threshold,
                                 int keep_all, cudaStream_t s) {
  const int64_t nwords = ((nbits + 7) / 8 + 3) / 4;
  int64_t blocks = (nwords + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  gen_keep_mask_kernel<<<int(blocks), 256, 0, s>>>(mask, nbits, seed, threshold, keep_all);
  return cudaGetLastError();
}

}  // namespace fav
