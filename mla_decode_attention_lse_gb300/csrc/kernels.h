// kernels.h -- host-side launch entry points of the kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "kparams.h"

namespace mla {

// CUDA-core kernel: any number of partials per token.
size_t simt_smem_bytes(int n_part);
cudaError_t launch_simt(const KParams &p, cudaStream_t stream);
// CUDA-core kernel for small batches (1 <= S <= 16, n_part <= 32): one CTA
// per (head, 16 V rows).
bool simt_small_fits(int S, int n_part);
size_t simt_small_smem_bytes();
int simt_small_grid(int H);
cudaError_t launch_simt_small(const KParams &p, cudaStream_t stream);

// Fused tcgen05 kernel: tile = 8, 16 or 32 tokens, n_part <= 32 (16 for 32-token tiles).
constexpr int kTcMaxPart = 32;
int tc_warps(int tile, int w_fmt, int n_part);        // warps per CTA
int tc_ctas_per_sm(int tile, int w_fmt, int n_part);  // resident CTAs per SM the grid is sized for
int tc_max_part(int tile, int w_fmt);                 // partials per token the tile supports
size_t tc_smem_bytes(int tile, int w_fmt, int n_part);
cudaError_t launch_tc(const KParams &p, int grid, cudaStream_t stream);

// Decode-size kernel: a (head, 16-token) unit per 4-CTA cluster, the latent
// dimension split over the cluster; n_part <= 16.
constexpr int kKsMaxPart = 16;
int ks_ctas_per_unit();
int ks_threads();
size_t ks_smem_bytes(int w_fmt);
cudaError_t launch_ks(const KParams &p, cudaStream_t stream);

// The DCP producer side: pack every rank's partials into one rank's buffer.
int pack_threads();
int pack_grid(long long rows, int num_sms);
cudaError_t launch_pack(const PackParams &p, int grid, cudaStream_t stream);

// The partial producer (split-KV MLA decode attention): one CTA per
// (request, split, head group) of q * G <= 32 query rows; the cache tensor
// [B, Lmax, 576] bf16 is read through `map` (boxes of 64 x 128 x 1, 128-byte
// swizzle).
int attn_heads_per_cta(int q, int H);  // G
int attn_rows(int q, int H);           // the MMA's N: q * G rounded up to 16
size_t attn_smem_bytes(int rows);
// Cached positions per tile of the attention kernel for `rows` query rows
// (the TMA box height of the cache tensor's map): 64 or 128.
int attn_tile_positions(int rows, bool fused);
cudaError_t launch_attn(const AttnParams &p, const CUtensorMap &map, int num_sms, cudaStream_t stream);
// The same attention on 2-CTA clusters: each CTA holds half of every cached
// row's latents (rank 1 also the rope part), the partial scores meet through
// distributed shared memory.
cudaError_t launch_attn_pair(const AttnParams &p, const CUtensorMap &map, int num_sms, cudaStream_t stream);
// The same attention with the combine of its partials behind it in the same
// launch (bf16 W_V through `wv_map`: [H, 128, 512], boxes of 64 x 128 x 1,
// 128-byte swizzle) and, when p.n_out > 0, the o_proj shard on its core rows
// (`wo_map`: W_o [n_out, H*128], `x_map`: core [S, H*128], both boxes of 64
// columns x 64 rows, 128-byte swizzle); p.ws holds 3 + attn_combine_tiles(S)
// zeroed words.
int attn_combine_tiles(int S);
cudaError_t launch_attn_combine(const AttnParams &p, const CUtensorMap &map, const CUtensorMap &wv_map,
                                const CUtensorMap &wo_map, const CUtensorMap &x_map, int num_sms, cudaStream_t stream);

}  // namespace mla
