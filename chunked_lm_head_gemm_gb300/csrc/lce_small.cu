// The small kernels of the path: label count, log-sum-exp combine, loss
// reduction, fp32 -> bf16 input conversion, the fused path's in-place
// exponentials -> gradient-logits pass and gradient scaling, and the
// bounded-wait probe.
#include "lce_device.cuh"

namespace lce {

// N = #{i : label i takes part}. Labels that are neither ignore_index nor in
// [0, V) raise the label-range bit and count as ignored, as everywhere else.
__global__ void k_count_valid(const int64_t* __restrict__ labels, int64_t L,
                              int64_t V, int64_t ignore_index,
                              unsigned long long* n_valid, unsigned* err) {
  unsigned long long c = 0;
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < L; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t y = labels[i];
    if (y != ignore_index) {
      if (y >= 0 && y < V)
        ++c;
      else
        bad = true;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
  const bool any_bad = __any_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0) {
    if (c) atomicAdd(n_valid, c);  // integer sum: order does not matter
    if (any_bad) atomicOr(err, ERRBIT_LABEL_RANGE);
  }
}

cudaError_t launch_count_valid(const int64_t* labels, int64_t L, int64_t V,
                               int64_t ignore_index,
                               unsigned long long* n_valid, unsigned* err,
                               cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(n_valid, 0, sizeof(unsigned long long), s);
  if (e != cudaSuccess) return e;
  const int64_t want = (L + 255) / 256;
  const int grid = static_cast<int>(want < 1024 ? (want < 1 ? 1 : want) : 1024);
  k_count_valid<<<grid, 256, 0, s>>>(labels, L, V, ignore_index, n_valid, err);
  return cudaGetLastError();
}

// lse_i = ln 2 * (M + log2 sum_k s_k 2^(m_k - M)), M = max_k m_k, merging the
// per-split partials in a fixed order; then a fixed-order block sum of the
// loss terms of the rows that take part, in float64: lse_i - z_i,y_i, or
// with a loss variant the smoothed cross entropy plus the z-loss,
// lse_i - (1 - eps) z_i,y_i - (eps / V) sum_j z_ij + zcoef lse_i^2 (the
// logit sums merged from part_z in split order).
constexpr int COMBINE_THREADS = COMBINE_ROWS;

__global__ void __launch_bounds__(COMBINE_THREADS)
    k_lse_combine(const float* __restrict__ part_m,
                  const float* __restrict__ part_s, int splits,
                  const float* __restrict__ zy,
                  const int64_t* __restrict__ labels, int64_t L, int64_t V,
                  int64_t ignore_index, float* __restrict__ lse,
                  double* __restrict__ block_sums,
                  const float* __restrict__ part_z, float eps, float zcoef) {
  __shared__ double warp_sums[COMBINE_THREADS / 32];
  const int64_t i = blockIdx.x * static_cast<int64_t>(COMBINE_THREADS) +
                    threadIdx.x;
  double term = 0.0;
  if (i < L) {
    float M = -INFINITY;
    for (int k = 0; k < splits; ++k) M = fmaxf(M, part_m[k * L + i]);
    float t = 0.f;
    for (int k = 0; k < splits; ++k)
      t += part_s[k * L + i] * exp2f(part_m[k * L + i] - M);
    const float l = (M + log2f(t)) * LN2;
    lse[i] = l;
    if (label_valid(labels[i], V, ignore_index)) {
      if (part_z == nullptr && zcoef == 0.f) {
        term = static_cast<double>(l) - static_cast<double>(zy[i]);
      } else {
        const double ld = static_cast<double>(l);
        double zsum = 0.0;
        if (part_z != nullptr)
          for (int k = 0; k < splits; ++k) zsum += part_z[k * L + i];
        const double e = static_cast<double>(eps);
        term = ld - (1.0 - e) * static_cast<double>(zy[i]) -
               e / static_cast<double>(V) * zsum +
               static_cast<double>(zcoef) * ld * ld;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) b += warp_sums[w];
    block_sums[blockIdx.x] = b;
  }
}

cudaError_t launch_lse_combine(const float* part_m, const float* part_s,
                               int splits, const float* zy,
                               const int64_t* labels, int64_t L, int64_t V,
                               int64_t ignore_index, float* lse,
                               double* block_sums, int* nblocks_out,
                               cudaStream_t s, const float* part_z, float eps,
                               float zcoef) {
  const int nb = static_cast<int>((L + COMBINE_THREADS - 1) / COMBINE_THREADS);
  *nblocks_out = nb;
  k_lse_combine<<<nb, COMBINE_THREADS, 0, s>>>(part_m, part_s, splits, zy,
                                               labels, L, V, ignore_index, lse,
                                               block_sums, part_z, eps, zcoef);
  return cudaGetLastError();
}

// Vocabulary slice [v0, v0 + Vs): per row, the split partials merged in
// split order into the slice's max logit m = ln 2 * M (natural units) and
// sum of exp(z - m) = sum_k s_k 2^(m_k - M); the label logit where the label
// lies in the slice, else 0 (so that summing the slices' values gives it);
// when part_z is set, the sum of the slice's logits (the split sums added in
// split order in float64, then rounded to float).
__global__ void __launch_bounds__(COMBINE_THREADS)
    k_slice_stats(const float* __restrict__ part_m,
                  const float* __restrict__ part_s, int splits,
                  const float* __restrict__ zy_in,
                  const int64_t* __restrict__ labels, int64_t L, int64_t v0,
                  int64_t Vs, int64_t V_total, int64_t ignore_index,
                  float* __restrict__ m, float* __restrict__ s,
                  float* __restrict__ zy, const float* __restrict__ part_z,
                  float* __restrict__ zsum) {
  const int64_t i = blockIdx.x * static_cast<int64_t>(COMBINE_THREADS) +
                    threadIdx.x;
  if (i >= L) return;
  float M = -INFINITY;
  for (int k = 0; k < splits; ++k) M = fmaxf(M, part_m[k * L + i]);
  float t = 0.f;
  for (int k = 0; k < splits; ++k)
    t += part_s[k * L + i] * exp2f(part_m[k * L + i] - M);
  m[i] = M * LN2;
  s[i] = t;
  const int64_t y = labels[i];
  const bool here = label_valid(y, V_total, ignore_index) && y >= v0 &&
                    y < v0 + Vs;
  zy[i] = here ? zy_in[i] : 0.f;
  if (part_z != nullptr) {
    double t = 0.0;
    for (int k = 0; k < splits; ++k) t += part_z[k * L + i];
    zsum[i] = static_cast<float>(t);
  }
}

cudaError_t launch_slice_stats(const float* part_m, const float* part_s,
                               int splits, const float* zy_in,
                               const int64_t* labels, int64_t L, int64_t v0,
                               int64_t Vs, int64_t V_total,
                               int64_t ignore_index, float* m, float* s_out,
                               float* zy, cudaStream_t s, const float* part_z,
                               float* zsum) {
  const int nb = static_cast<int>((L + COMBINE_THREADS - 1) / COMBINE_THREADS);
  k_slice_stats<<<nb, COMBINE_THREADS, 0, s>>>(part_m, part_s, splits, zy_in,
                                               labels, L, v0, Vs, V_total,
                                               ignore_index, m, s_out, zy,
                                               part_z, zsum);
  return cudaGetLastError();
}

// P vocabulary slices' (m, s, zy), each [P][L]: lse = M + ln sum_r s_r
// exp(m_r - M) with M = max_r m_r, the label logit = sum_r zy_r, merged in
// slice order; then per-256-row float64 sums of (lse - z_y) over rows that
// take part, as k_lse_combine. With a loss variant (zsum set or zcoef != 0)
// the term is lse - (1 - eps) z_y - (eps / V_total) sum_r zsum_r + zcoef
// lse^2, the slices' logit sums added in slice order in float64.
__global__ void __launch_bounds__(COMBINE_THREADS)
    k_combine_slices(const float* __restrict__ m, const float* __restrict__ s,
                     const float* __restrict__ zy, int64_t P,
                     const int64_t* __restrict__ labels, int64_t L,
                     int64_t V_total, int64_t ignore_index,
                     float* __restrict__ lse,
                     double* __restrict__ block_sums,
                     const float* __restrict__ zsum, float eps, float zcoef) {
  __shared__ double warp_sums[COMBINE_THREADS / 32];
  const int64_t i = blockIdx.x * static_cast<int64_t>(COMBINE_THREADS) +
                    threadIdx.x;
  double term = 0.0;
  if (i < L) {
    float M = -INFINITY;
    for (int64_t r = 0; r < P; ++r) M = fmaxf(M, m[r * L + i]);
    float t = 0.f, z = 0.f;
    for (int64_t r = 0; r < P; ++r) {
      t += s[r * L + i] * exp2f((m[r * L + i] - M) * LOG2E);
      z += zy[r * L + i];
    }
    const float l = M + log2f(t) * LN2;
    lse[i] = l;
    if (label_valid(labels[i], V_total, ignore_index)) {
      if (zsum == nullptr && zcoef == 0.f) {
        term = static_cast<double>(l) - static_cast<double>(z);
      } else {
        const double ld = static_cast<double>(l);
        double zs = 0.0;
        if (zsum != nullptr)
          for (int64_t r = 0; r < P; ++r) zs += zsum[r * L + i];
        const double e = static_cast<double>(eps);
        term = ld - (1.0 - e) * static_cast<double>(z) -
               e / static_cast<double>(V_total) * zs +
               static_cast<double>(zcoef) * ld * ld;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = term;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) b += warp_sums[w];
    block_sums[blockIdx.x] = b;
  }
}

cudaError_t launch_combine_slices(const float* m, const float* s_in,
                                  const float* zy, int64_t P,
                                  const int64_t* labels, int64_t L,
                                  int64_t V_total, int64_t ignore_index,
                                  float* lse, double* block_sums,
                                  int* nblocks_out, cudaStream_t s,
                                  const float* zsum, float eps, float zcoef) {
  const int nb = static_cast<int>((L + COMBINE_THREADS - 1) / COMBINE_THREADS);
  *nblocks_out = nb;
  k_combine_slices<<<nb, COMBINE_THREADS, 0, s>>>(m, s_in, zy, P, labels, L,
                                                  V_total, ignore_index, lse,
                                                  block_sums, zsum, eps,
                                                  zcoef);
  return cudaGetLastError();
}

// loss = (sum of block sums, fixed order) / N, and 0 when N = 0.
__global__ void __launch_bounds__(256)
    k_loss_finalize(const double* __restrict__ block_sums, int nblocks,
                    const unsigned long long* __restrict__ n_valid,
                    float* __restrict__ loss) {
  __shared__ double part[256];
  double acc = 0.0;
  for (int b = threadIdx.x; b < nblocks; b += 256) acc += block_sums[b];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const unsigned long long n = *n_valid;
    *loss = n ? static_cast<float>(part[0] / static_cast<double>(n)) : 0.f;
  }
}

cudaError_t launch_loss_finalize(const double* block_sums, int nblocks,
                                 const unsigned long long* n_valid,
                                 float* loss, cudaStream_t s) {
  k_loss_finalize<<<1, 256, 0, s>>>(block_sums, nblocks, n_valid, loss);
  return cudaGetLastError();
}

// fp32 -> bf16 (round to nearest even), 8 elements per thread when aligned.
__global__ void k_f32_to_bf16(const float* __restrict__ in,
                              uint16_t* __restrict__ out, int64_t n) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < n; i += stride)
    out[i] = to_bf16_bits(in[i]);
}

cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n,
                               cudaStream_t s) {
  const int64_t want = (n + 255) / 256;
  const int grid = static_cast<int>(want < 4096 ? (want < 1 ? 1 : want) : 4096);
  k_f32_to_bf16<<<grid, 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

// In place over one row chunk of the fused forward+backward: E holds
// e = 2^(u - m_t) (bf16), u = z log2 e, m_t the maximum of u over the
// 256-column tile; with lse2 = lse log2 e the softmax is e 2^(m_t - lse2),
// so G = e 2^(m_t - lse2) - [j == y] on rows that take part, 0 elsewhere;
// with a loss variant G = zf e 2^(m_t - lse2) - ome [j == y] - eps_v
// (VariantGrad; zf folded into the scale sc).
// Works on 16-byte vectors of 8 consecutive columns (8 divides the
// 256-column tile, so a vector never straddles two tiles). Columns between
// V and ldg are padding that nothing reads.
__device__ __forceinline__ uint4 exp_to_grad(uint4 in, float sc, int yo,
                                             float ome, float eps_v) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float lo = fmaf(__uint_as_float(w[q] << 16), sc, -eps_v);
    float hi = fmaf(__uint_as_float(w[q] & 0xFFFF0000u), sc, -eps_v);
    if (2 * q == yo) lo -= ome;
    if (2 * q + 1 == yo) hi -= ome;
    o[q] = pack_bf16x2(lo, hi);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The chunk's rows x ceil(V/8) 16-byte vectors are cut into one contiguous
// range per block (so every block moves the same bytes, whatever the row
// count), walked row segment by row segment; each thread keeps GFE_U vectors
// in flight. Rows that do not take part are zeroed without being read.
constexpr int GFE_THREADS = 256;
constexpr int GFE_BLOCKS_PER_SM = 4;
constexpr int GFE_U = 8;

__global__ void __launch_bounds__(GFE_THREADS, GFE_BLOCKS_PER_SM)
    k_grad_from_exp(uint16_t* __restrict__ E, int64_t ldg,
                    const float* __restrict__ tile_max, int64_t num_n,
                    const float* __restrict__ lse,
                    const int64_t* __restrict__ labels, int64_t rows,
                    int64_t V, int64_t ignore_index, int64_t slice_v0,
                    int64_t v_total, VariantGrad var) {
  const int64_t nvec = (V + 7) / 8;
  const int64_t vt = v_total > 0 ? v_total : V;
  const int64_t total = rows * nvec;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  int64_t pos = static_cast<int64_t>(blockIdx.x) * per;
  const int64_t end = pos + per < total ? pos + per : total;
  while (pos < end) {
    const int64_t row = pos / nvec;
    const int64_t vb = pos - row * nvec;
    const int64_t ve = (end - pos < nvec - vb) ? vb + (end - pos) : nvec;
    pos += ve - vb;
    const int64_t y = labels[row];
    uint4* er = reinterpret_cast<uint4*>(E + row * ldg);
    if (!label_valid(y, vt, ignore_index)) {
      for (int64_t v = vb + threadIdx.x; v < ve; v += GFE_THREADS)
        er[v] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const float l2 = lse[row] * LOG2E;
    const float zf = fmaf(var.zloss2, lse[row], 1.f);
    const float* tm = tile_max + row * num_n;
    // the label's column in this slice, or far below any column
    const int64_t yl = y - slice_v0;
    const int ycol = (yl >= 0 && yl < V) ? static_cast<int>(yl) : -(1 << 30);
    for (int64_t v0 = vb + threadIdx.x; v0 < ve;
         v0 += static_cast<int64_t>(GFE_U) * GFE_THREADS) {
      uint4 in[GFE_U];
#pragma unroll
      for (int k = 0; k < GFE_U; ++k) {
        const int64_t v = v0 + static_cast<int64_t>(k) * GFE_THREADS;
        if (v < ve) in[k] = er[v];
      }
#pragma unroll
      for (int k = 0; k < GFE_U; ++k) {
        const int64_t v = v0 + static_cast<int64_t>(k) * GFE_THREADS;
        if (v < ve) {
          const int64_t j0 = v * 8;
          er[v] = exp_to_grad(in[k], ex2(tm[j0 >> 8] - l2) * zf,
                              ycol - static_cast<int>(j0), var.ome,
                              var.eps_v);
        }
      }
    }
  }
}

cudaError_t launch_grad_from_exp(uint16_t* E, int64_t ldg,
                                 const float* tile_max, int64_t num_n,
                                 const float* lse, const int64_t* labels,
                                 int64_t rows, int64_t V, int64_t ignore_index,
                                 int num_sms, cudaStream_t s, int64_t v0,
                                 int64_t v_total, VariantGrad var) {
  const int64_t work = rows * ((V + 7) / 8);
  const int64_t full = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) *
                       GFE_BLOCKS_PER_SM;
  const int64_t want = (work + GFE_THREADS - 1) / GFE_THREADS;
  const unsigned grid =
      static_cast<unsigned>(want < full ? (want < 1 ? 1 : want) : full);
  k_grad_from_exp<<<grid, GFE_THREADS, 0, s>>>(E, ldg, tile_max, num_n, lse,
                                               labels, rows, V, ignore_index,
                                               v0, v_total, var);
  return cudaGetLastError();
}

// dH *= d and dW *= d with d = dloss[0]; nothing to do when d == 1.
// n_dh is a multiple of 8 (bf16) or 4 (fp32), n_dw a multiple of 4 (H is a
// multiple of 8), so every access is a 16-byte vector.
__global__ void k_scale_grads(void* __restrict__ dH, int dh_f32, int64_t n_dh,
                              float* __restrict__ dW, int64_t n_dw,
                              const float* __restrict__ dloss) {
  const float d = *dloss;
  if (d == 1.f) return;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (dh_f32) {
    float4* p = static_cast<float4*>(dH);
    for (int64_t i = t0; i < n_dh / 4; i += stride) {
      float4 x = p[i];
      x.x *= d; x.y *= d; x.z *= d; x.w *= d;
      p[i] = x;
    }
  } else {
    uint4* p = static_cast<uint4*>(dH);
    for (int64_t i = t0; i < n_dh / 8; i += stride) {
      const uint4 x = p[i];
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        o[q] = pack_bf16x2(__uint_as_float(w[q] << 16) * d,
                           __uint_as_float(w[q] & 0xFFFF0000u) * d);
      p[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  float4* q4 = reinterpret_cast<float4*>(dW);
  for (int64_t i = t0; i < n_dw / 4; i += stride) {
    float4 x = q4[i];
    x.x *= d; x.y *= d; x.z *= d; x.w *= d;
    q4[i] = x;
  }
}

cudaError_t launch_scale_grads(void* dH, int dh_f32, int64_t n_dh, float* dW,
                               int64_t n_dw, const float* dloss,
                               cudaStream_t s) {
  k_scale_grads<<<1024, 256, 0, s>>>(dH, dh_f32, n_dh, dW, n_dw, dloss);
  return cudaGetLastError();
}

// Row-sharded sequences: one shard's share of the sequence's loss for the
// caller's sum over the shards, sums = (N_r loss_r, N_r) in float64; and,
// from the summed pair (S, N), the sequence's loss S / N and this shard's
// gradient weight dloss N_r / N, both 0 when N = 0 (a NULL dloss is 1).
__global__ void k_shard_sums(const float* __restrict__ loss_local,
                             const unsigned long long* __restrict__ n_local,
                             double* __restrict__ sums) {
  const double n = static_cast<double>(*n_local);
  sums[0] = n * static_cast<double>(*loss_local);
  sums[1] = n;
}

__global__ void k_combine_shards(const double* __restrict__ sums,
                                 const unsigned long long* __restrict__ n_local,
                                 const float* __restrict__ dloss,
                                 float* __restrict__ loss,
                                 float* __restrict__ weight) {
  const double n = sums[1];
  const double d = dloss != nullptr ? static_cast<double>(*dloss) : 1.0;
  *loss = n > 0.0 ? static_cast<float>(sums[0] / n) : 0.f;
  *weight = n > 0.0 ? static_cast<float>(d * static_cast<double>(*n_local) / n)
                    : 0.f;
}

cudaError_t launch_shard_sums(const float* loss_local,
                              const unsigned long long* n_local, double* sums,
                              cudaStream_t s) {
  k_shard_sums<<<1, 1, 0, s>>>(loss_local, n_local, sums);
  return cudaGetLastError();
}

cudaError_t launch_combine_shards(const double* sums,
                                  const unsigned long long* n_local,
                                  const float* dloss, float* loss,
                                  float* weight, cudaStream_t s) {
  k_combine_shards<<<1, 1, 0, s>>>(sums, n_local, dloss, loss, weight);
  return cudaGetLastError();
}

// One thread waits on an mbarrier that nothing arrives at, with the same
// bounded wait the contraction kernels use; it must give up after
// timeout_ns and raise the timeout bit. Used to test failure detection
// without hanging the GPU.
__global__ void k_wait_probe(unsigned* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const WaitCtx ctx{&abort_flag, err, timeout_ns};
    mbar_wait(smem_u32(&bar), 0, ctx, true);
  }
}

cudaError_t launch_wait_probe(unsigned* err, uint64_t timeout_ns,
                              cudaStream_t s) {
  k_wait_probe<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lce
