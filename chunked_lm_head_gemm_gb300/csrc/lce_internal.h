// Internal declarations shared by the host layer and the kernel translation
// units of the fused linear cross-entropy library. Not part of the C-ABI.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace lce {

// Tile shape of every tensor-core contraction: one CTA owns a 128 x 256 fp32
// accumulator in tensor memory and walks K in steps of 64 bf16 elements
// (one 128-byte swizzle row).
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int GEMM_THREADS = 192;           // 6 warps: TMA, MMA, 4 x epilogue
// Epilogue staging for TMA stores: per epilogue warp two buffers of one
// EPI_BOX x EPI_BOX bf16 box (32 rows x 64 bytes), after the barriers.
constexpr int EPI_BOX = 32;
constexpr int EPI_BUF_BYTES = EPI_BOX * EPI_BOX * 2;     // 2 KB
constexpr int EPI_STAGE_BYTES = 4 * 2 * EPI_BUF_BYTES;  // 16 KB
constexpr int GEMM_SMEM_BYTES =
    1024 + STAGES * STAGE_BYTES + 1024 + EPI_STAGE_BYTES;
constexpr int TMEM_COLS = 512;              // two 256-column accumulators

// Rows per block of the per-row combine kernels (one float64 loss sum per
// block).
constexpr int COMBINE_ROWS = 256;

// Device error bits, OR-ed into the library's error word.
constexpr unsigned ERRBIT_LABEL_RANGE = 1u << 4;
constexpr unsigned ERRBIT_TIMEOUT = 1u << 5;

// Work decomposition of one contraction D[M,N] = A[M,K] B[K,N].
// A unit is (row block m_blk, a run of n_count consecutive column tiles
// starting at n_first). Units are numbered u = m_blk * splits + split.
struct GemmGeom {
  int64_t M, N, K;
  int num_m, num_n, num_kb;
  int splits;           // column-tile runs per row block
  int tiles_per_split;  // column tiles per run (the last run may be shorter)
  int num_units;        // num_m * splits
  uint64_t timeout_ns;  // limit of every wait inside the kernel
  // Tile order when every unit is one tile (splits == num_n): 0 = row
  // block major; g > 0 = groups of g column tiles, row blocks inside a
  // group (a wave then touches fewer column panels).
  int group_n;
  // B from two tensor maps: 0 = one map; 1 = along N, each 256-row B tile
  // being 128 rows of the first map then the same 128 rows of the second
  // (tiles then cover 128 output columns, num_n = ceil(N / 128)); 2 = along
  // K, k-blocks from k_split_kb on read the second map (at k - k_split_kb).
  int b_dual;
  int k_split_kb;
  // Wave pacing (nullptr: off): before its s-th output tile (s >= 1) a
  // CTA's (a pair's leader's) producer waits until *wave_ctr >= s * (CTAs or
  // clusters of the grid), i.e. until every CTA has issued the loads of s
  // tiles, for at most wave_wait_ns; after issuing a tile's loads it adds 1,
  // and when done it adds wave_steps minus its tile count (wave_steps = the
  // most tiles any CTA has), so finished CTAs hold no one back. Keeps the
  // CTAs that share operand panels at the same K position so the panels
  // are read from L2, not DRAM. Only a hint: a wait that runs out goes on.
  // The counter is zeroed before every launch.
  unsigned* wave_ctr;
  uint32_t wave_wait_ns;
  uint32_t wave_steps;
};

// ---- epilogue parameter blocks ----------------------------------------------

// Forward logits tile -> per-row online (max, sum of exp) over the unit's
// columns, plus the logit at the label.
// Vocabulary slices (v0, v_total; both 0 for the whole vocabulary): the
// contraction's N columns are the vocabulary ids [v0, v0 + N) of a
// vocabulary of v_total; a row takes part when its label is a valid id of
// the whole vocabulary, and its label column is y - v0 when that lies in
// the slice.
struct LseParams {
  const int64_t* labels;  // [M]
  float* part_m;          // [splits][M], running max in log2 units
  float* part_s;          // [splits][M], sum of 2^(u - max)
  float* zy;              // [M], logit at the label (rows whose label is here)
  int64_t ignore_index;
  int64_t v0, v_total;
  float* part_z;          // [splits][M], sum of the logits (label smoothing),
                          // or NULL
};

// The loss variants' constants for the gradient logits (all rows that take
// part): G = zf_i softmax - ome [j == y] - eps_v with zf_i = 1 + zloss2 lse_i,
// i.e. zloss2 = 2 * z-loss coefficient, ome = 1 - label smoothing, eps_v =
// label smoothing / V. The plain loss is {0, 1, 0}, whose arithmetic gives
// the plain gradient's bits exactly.
struct VariantGrad {
  float zloss2;
  float ome;
  float eps_v;
};

// Backward recompute tile -> G = softmax - onehot (unscaled), bf16.
struct GradParams {
  const int64_t* labels;  // [M], rows of this chunk
  const float* lse;       // [M], rows of this chunk
  uint16_t* G;            // [M][ldg] bf16 bits (the kernel writes it through
                          // the store map launched with it, not this pointer)
  int64_t ldg;
  int64_t ignore_index;
  int64_t v0, v_total;    // vocabulary slice, as LseParams
  VariantGrad var;        // loss variant ({0, 1, 0}: plain)
};

// Fused forward+backward, logits of one row chunk -> per-split online
// (max, sum) partials and the label logit (as LseParams), plus each tile's
// row maximum and the tile's exponentials e = 2^(u - tile max) in bf16,
// which a later pass rescales into the gradient logits in place.
struct FusedParams {
  const int64_t* labels;  // [M], rows of this chunk
  float* part_m;          // [splits][M]
  float* part_s;          // [splits][M]
  float* zy;              // [M]
  uint16_t* E;            // [M][ldg] bf16 bits (written through the store
                          // map launched with the kernel)
  int64_t ldg;
  float* tile_max;        // [M][num_n], log2 units
  int64_t ignore_index;
  int64_t v0, v_total;    // vocabulary slice, as LseParams
  float* part_z;          // [splits][M] logit sums, or NULL (as LseParams)
};

// Gated-MLP gate/up contraction (B dual along N): accumulator columns
// 0..127 hold g, 128..255 hold u for output columns [128 n, 128 n + 128);
// writes a = silu(g) * u and, when asked, g and u (bf16), each through its
// store map (32 x 32 boxes, as the logits epilogues' chunks). The maps
// reach the kernel inside this block, a __grid_constant__ parameter.
struct SwigluParams {
  CUtensorMap map_a;      // store map of a [M][I]
  CUtensorMap map_g;      // of g [M][I] (used when save_gu)
  CUtensorMap map_u;      // of u [M][I] (used when save_gu)
  int save_gu;
};

// Gated-MLP backward: the accumulator is da = dy Wd; with the saved g, u
// writes dg = da u silu'(g) at [row][col] and du = da silu(g) at
// [row][du_off + col] (bf16) through one store map of [dg | du].
struct SwigluBwdParams {
  CUtensorMap map_dgu;    // store map of dgu [M][2 I]
  const uint16_t* g;      // [M][ld_gu]
  const uint16_t* u;      // [M][ld_gu]
  int64_t ld_gu;
  int64_t du_off;
};

// Plain store of scale * acc (dH chunk, or the building-block test GEMM).
struct StoreParams {
  void* out;              // [M][ldo]
  int64_t ldo;
  void* out2;             // rows >= split_row go to out2 (row - split_row),
  int64_t split_row;      // when out2 is not NULL
  int out_f32;            // 1: fp32 output, 0: bf16 output
  int accumulate;         // 1: out += scale*acc (fp32 only), 0: out = scale*acc
  const float* dloss;     // scale = dloss[0] / n_valid[0] (n_valid 0 -> 0);
  const unsigned long long* n_valid;  // dloss NULL counts as 1, n_valid
                                      // NULL as 1: both NULL -> scale = 1
};

// ---- launch wrappers (defined in the kernel translation units) --------------
// Each launches one persistent tensor-core contraction on `stream`.
// a_mn / b_mn: operand stored MN-major (true) or K-major (false).
cudaError_t launch_gemm_lse(const CUtensorMap& ta, const CUtensorMap& tb,
                            const GemmGeom& g, const LseParams& p,
                            unsigned* err, int grid, cudaStream_t s);
// The gated-MLP contractions (gate/up with the SwiGLU epilogue, and da
// with the SwiGLU backward epilogue); tb2 is the second B map (b_dual).
cudaError_t launch_gemm_swiglu(bool pair, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tb2,
                               const GemmGeom& g, const SwigluParams& p,
                               unsigned* err, int grid, cudaStream_t s);
cudaError_t launch_gemm_swiglu_bwd(bool pair, const CUtensorMap& ta,
                                   const CUtensorMap& tb,
                                   const CUtensorMap& tb2, const GemmGeom& g,
                                   const SwigluBwdParams& p, unsigned* err,
                                   int grid, cudaStream_t s);

cudaError_t launch_gemm_grad(const CUtensorMap& ta, const CUtensorMap& tb,
                             const CUtensorMap& tg,
                             const GemmGeom& g, const GradParams& p,
                             unsigned* err, int grid, cudaStream_t s);
cudaError_t launch_gemm_fused(const CUtensorMap& ta, const CUtensorMap& tb,
                              const CUtensorMap& te,
                              const GemmGeom& g, const FusedParams& p,
                              unsigned* err, int grid, cudaStream_t s);
cudaError_t launch_gemm_store(bool a_mn, bool b_mn, const CUtensorMap& ta,
                              const CUtensorMap& tb, const GemmGeom& g,
                              const StoreParams& p, unsigned* err, int grid,
                              cudaStream_t s,
                              const CUtensorMap* tb2 = nullptr);

// The same four contractions on CTA pairs (cluster of 2, tcgen05
// cta_group::2, 256 x 256 tiles): geometry in units of 256 rows, grid even,
// K-major B boxes of 128 rows.
cudaError_t launch_gemm_pair_lse(const CUtensorMap& ta, const CUtensorMap& tb,
                                 const GemmGeom& g, const LseParams& p,
                                 unsigned* err, int grid, cudaStream_t s);
cudaError_t launch_gemm_pair_grad(const CUtensorMap& ta, const CUtensorMap& tb,
                                  const CUtensorMap& tg,
                                  const GemmGeom& g, const GradParams& p,
                                  unsigned* err, int grid, cudaStream_t s);
cudaError_t launch_gemm_pair_fused(const CUtensorMap& ta,
                                   const CUtensorMap& tb,
                                   const CUtensorMap& te, const GemmGeom& g,
                                   const FusedParams& p, unsigned* err,
                                   int grid, cudaStream_t s);
cudaError_t launch_gemm_pair_store(bool a_mn, bool b_mn, const CUtensorMap& ta,
                                   const CUtensorMap& tb, const GemmGeom& g,
                                   const StoreParams& p, unsigned* err,
                                   int grid, cudaStream_t s,
                                   const CUtensorMap* tb2 = nullptr);

// How many CTA pairs of the contraction kernels can be resident at once
// (clusters are placed within a GPC, so this can be below SMs / 2).
cudaError_t pair_max_active_clusters(int* n);

// Small kernels.
cudaError_t launch_count_valid(const int64_t* labels, int64_t L, int64_t V,
                               int64_t ignore_index,
                               unsigned long long* n_valid, unsigned* err,
                               cudaStream_t s);
// lse per row from the split partials, and per-256-row float64 sums of the
// loss terms of the rows that take part: lse - z_y for the plain loss; with
// a variant (part_z set or zcoef != 0) lse - (1 - eps) z_y - (eps / V)
// sum_j z_j + zcoef lse^2, the logit sums merged from part_z in split order.
cudaError_t launch_lse_combine(const float* part_m, const float* part_s,
                               int splits, const float* zy,
                               const int64_t* labels, int64_t L, int64_t V,
                               int64_t ignore_index, float* lse,
                               double* block_sums, int* nblocks_out,
                               cudaStream_t s, const float* part_z = nullptr,
                               float eps = 0.f, float zcoef = 0.f);
// Vocabulary slice: merge the per-split partials into the slice's per-row
// max logit m (natural units) and sum of exp(z - m), and the label logit
// (0 where the label is not in [v0, v0 + Vs)); with part_z, also the
// slice's per-row logit sum zsum.
cudaError_t launch_slice_stats(const float* part_m, const float* part_s,
                               int splits, const float* zy_in,
                               const int64_t* labels, int64_t L, int64_t v0,
                               int64_t Vs, int64_t V_total,
                               int64_t ignore_index, float* m, float* s_out,
                               float* zy, cudaStream_t s,
                               const float* part_z = nullptr,
                               float* zsum = nullptr);
// P slices' statistics ([P][L] each) -> lse and per-256-row loss sums, the
// slices merged in slice order; a loss variant as launch_lse_combine, the
// logit sums from the slices' zsum ([P][L]).
cudaError_t launch_combine_slices(const float* m, const float* s_in,
                                  const float* zy, int64_t P,
                                  const int64_t* labels, int64_t L,
                                  int64_t V_total, int64_t ignore_index,
                                  float* lse, double* block_sums,
                                  int* nblocks_out, cudaStream_t s,
                                  const float* zsum = nullptr, float eps = 0.f,
                                  float zcoef = 0.f);
cudaError_t launch_loss_finalize(const double* block_sums, int nblocks,
                                 const unsigned long long* n_valid,
                                 float* loss, cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float* in, uint16_t* out, int64_t n,
                               cudaStream_t s);
// In place over one row chunk: E[i][j] = 2^(u - tile max) becomes
// G = 2^(tile max - lse_i log2 e) E - [j == y_i] (bf16), 0 on ignored rows;
// with a loss variant, G = zf_i 2^(tile max - lse_i log2 e) E - ome [j ==
// y_i] - eps_v (VariantGrad).
// For a vocabulary slice (v0, v_total as LseParams) the onehot sits at
// column y_i - v0 and validity is judged against v_total.
cudaError_t launch_grad_from_exp(uint16_t* E, int64_t ldg,
                                 const float* tile_max, int64_t num_n,
                                 const float* lse, const int64_t* labels,
                                 int64_t rows, int64_t V, int64_t ignore_index,
                                 int num_sms, cudaStream_t s,
                                 int64_t v0 = 0, int64_t v_total = 0,
                                 VariantGrad var = VariantGrad{0.f, 1.f, 0.f});
// dH *= dloss[0] (bf16 or fp32) and dW *= dloss[0], skipped when dloss is 1.
cudaError_t launch_scale_grads(void* dH, int dh_f32, int64_t n_dh, float* dW,
                               int64_t n_dw, const float* dloss,
                               cudaStream_t s);
cudaError_t launch_wait_probe(unsigned* err, uint64_t timeout_ns,
                              cudaStream_t s);
// Row-sharded sequences: sums = (N_r loss_r, N_r) in float64; from the
// shards' summed pair, the sequence's loss and this shard's gradient weight.
cudaError_t launch_shard_sums(const float* loss_local,
                              const unsigned long long* n_local, double* sums,
                              cudaStream_t s);
cudaError_t launch_combine_shards(const double* sums,
                                  const unsigned long long* n_local,
                                  const float* dloss, float* loss,
                                  float* weight, cudaStream_t s);

}  // namespace lce
