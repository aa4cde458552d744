// Argument blocks and entry points of the packed CTC kernels (internal).
#pragma once

#include "ctc_common.cuh"

namespace ctcp {

struct PrepArgs {
    Layout L;
    void* ws;
    const int32_t* cu;
    const int32_t* lengths;
    const int32_t* target_lengths;
    float* loss;
    int reduction;
    int zero_infinity;
    int need_grad;
    int group_pairs;  // pairs one chain warp owns: longer targets run on a whole CTA
    int logits;       // the input rows are logits (log_softmax is taken by the path)
    int ckpt;         // state rows kept: every one (1) or those at multiples of ckpt
};

struct ChainArgs {
    Layout L;
    void* ws;
    const void* lp;      // (T_total, D) log probabilities
    int64_t lp_bytes;    // T_total * D * element bytes
    const int32_t* cu;   // cu_seqlens
    const int32_t* targets;
    const int32_t* target_lengths;
    float* loss;
    int D;
    int blank;
    int reduction;
    int zero_infinity;
    const float* lse;    // per-row log-sum-exp of logits input, subtracted from each value; null for log probabilities
    int store_rows;      // state rows kept for the backward: 0 none (loss only), 1 every row,
                         // K > 1 (a power of two) only rows whose index is a multiple of K
};

struct GradArgs {
    Layout L;
    void* ws;
    const void* lp;
    void* grad;
    const int32_t* cu;
    const int32_t* targets;
    const float* grad_loss;
    int D;
    int blank;
    int reduction;
    int zero_infinity;
    int rows_per_tile;   // rows per warp group
    int64_t n_tiles;     // warp groups
    int entry_cap;       // corrections a group can hold
    size_t warp_smem;    // shared memory bytes per warp
    int congruent;       // lp and grad share their address modulo 16
    uint32_t gp_mul;     // offset group of pair j: (j * gp_mul) >> 21 == j / L.gpairs
    int ckpt;            // the forward's checkpoint interval (1: every state row was stored)
};

// The gradient stream for wide rows (stream.cu): class sums and dense rows in
// one pass, fed by bulk copies into per-team shared-memory slots.
struct StreamArgs {
    Layout L;
    void* ws;
    const void* lp;
    void* grad;
    const int32_t* cu;  // cu_seqlens
    const int32_t* targets;
    const float* grad_loss;
    int D;
    int blank;
    int reduction;
    int zero_infinity;
    int elem_bytes;
    uint32_t gp_mul;    // offset group of pair j: (j * gp_mul) >> 21 == j / L.gpairs
    int nteams, nslots; // teams (a producer warp and four worker warps) per CTA, shared-memory slots per team
    int team_bytes;     // shared memory of one team
    int lp_cap, sr_cap, slot_bytes;  // a slot: lp span, stored alpha row, stored beta row, label records
    int desc_off, mbar_off, slots_off, ecls_off, eval_off, labm_off, labe_off, blkm_off, blke_off, red_off;
};

__global__ void prep_kernel(PrepArgs a);
template <int DT>
__global__ void lse_kernel(ChainArgs a);
template <int DT>
__global__ void emit_kernel(ChainArgs a);
template <int P, int G, int MAXT, bool CKPT>
__global__ void chain_kernel(ChainArgs a);
__global__ void post_kernel(GradArgs a);
template <int DT>
__global__ void grad_kernel(GradArgs a);
template <int DT>
__global__ void stream_kernel(StreamArgs a);
bool stream_plan(StreamArgs& a);  // team count and slot layout; false when one team does not fit
void grad_geometry(const Layout& L, int D, int& rows, int& entry_cap, size_t& warp_smem);
uint32_t grad_group_multiplier(const Layout& L);  // 0 if no exact multiplier exists

// Host launchers (defined next to their kernels).
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_lse(const ChainArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_emit(const ChainArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_chain(const ChainArgs& a, cudaStream_t s);
cudaError_t launch_post(const GradArgs& a, cudaStream_t s);
cudaError_t launch_grad(const GradArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_stream(const StreamArgs& a, int dtype, cudaStream_t s);
__global__ void segpost_kernel(GradArgs a);
cudaError_t launch_segpost(const GradArgs& a, cudaStream_t s);
int segpost_max_ckpt(const Layout& L);  // largest checkpoint interval the recompute supports (0: none)
// Workspace of the float64 path (f64.cu): the whole layout, or its loss-only prefix.
size_t f64_workspace_bytes(int64_t T_total, int32_t B, int32_t max_target_len, int32_t D, bool loss_only);

}  // namespace ctcp
