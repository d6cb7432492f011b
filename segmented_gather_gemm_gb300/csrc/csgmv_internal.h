// Internal interface between the C-ABI layer (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/csgmv.h"

namespace csgmv {

constexpr int kMinChunkSize = 16;  // chunked_backend.py MIN_CHUNK_SIZE
constexpr int kMaxRank = 64;       // largest buffer rank R the LoRA kernels take
constexpr int kMaxSlices = 3;
constexpr int kWideCols = 32768;   // output columns from which 16- / 32-token csgmv_qkv calls split
constexpr int kMaxKParts = 4;      // fp32 h planes of the csgmv_qkv workspace (parts of K)
constexpr size_t kWsHeader = 256;  // bytes before the planes: the part count the shrink chose
constexpr int kDecMaxParts = 32;   // planes of the decode kernels' split-K shrink
constexpr int kDecTM = 64;         // tokens of one decode tile at most (the batch info's tile table)
constexpr int kDecPermCap = 2048;  // tokens of a batch the decode kernels take

#ifdef __CUDACC__
// Programmatic dependent launch.  A kernel launched with
// cudaLaunchAttributeProgrammaticStreamSerialization may start while the
// kernel before it in the stream is still running; it calls griddep_wait()
// before its first access to global memory, which returns once that kernel
// has finished and its writes are visible (at once after a normal launch).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
// Lets a kernel launched next with that attribute start launching now; it
// still waits for this kernel's completion in griddep_wait().
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
#endif

enum LoraMode { kModeFused = 0, kModeShrink = 1, kModeExpand = 2 };

// Everything one launch of the shrink / expand / fused kernel needs.  Batch
// info arrays are read on the device, so a captured graph follows whatever
// batch was built into them last.
struct LoraParams {
    const uint16_t *x;   // (s, K) bf16
    const uint16_t *A;   // (max_loras, c*R, K) bf16
    const uint16_t *B;   // (max_loras, N, R) bf16
    // B of slice j as its own tensor: rows w * b_rows[j] + b_row0[j] + (n - off[j])
    // of Bs[j] (R bf16 each) hold B[w][n] for n in slice j.  One (L, N, R)
    // tensor is Bs[j] = B, b_rows[j] = N, b_row0[j] = off[j].
    const uint16_t *Bs[kMaxSlices];
    int b_rows[kMaxSlices], b_row0[kMaxSlices];
    int b_tuple;         // 1: the slices are separate tensors (slice offsets multiples of 64)
    uint16_t *y;         // (s, N) bf16, in/out
    void *h;             // (s, ldh) bf16 or f32 (shrink output / expand input)
    int64_t K, N, ldh;
    // fp32 h held as h_parts partial sums over parts of K, h_plane elements
    // apart (the csgmv_qkv workspace path); 1 = h itself
    int h_parts;
    int64_t h_plane;
    const int *h_parts_dev;  // the part count as the shrink chose it (read on the device, <= h_parts), or NULL
    int h_f32;
    int c, R;
    int off[kMaxSlices + 1];
    int accumulate;
    int num_tokens;      // s, bound for permutation entries
    int max_loras;
    int nsplit;          // column blocks per token tile (fused / expand)
    const int32_t *seg_indptr, *weight_indices, *permutation, *lora_ranks;
    const float *scalings;
    const int32_t *num_segments_dev, *max_len_dev;
    const int32_t *tile_table;  // the batch info's decode tiles, or NULL
    int32_t *status;
    // shared-memory carve-up (bytes from the dynamic base), chosen on the host
    int sm_tok, sm_stage, sm_hpart, sm_hred, sm_hbf, sm_ex;
    int shrink_stage_bytes, ex_stage_bytes, ex_stages;
    int hrow_pitch;      // floats per row of hpart / hred
    int rows_per_rank;   // TM / cluster size (reduce-scatter rows per CTA)
    int ex_prefetch;     // 1: expand stages do not alias the shrink stages
};

struct LaunchInfo {
    int tm;              // token tile
    int crmax;           // compile-time bound on c*R
    int cluster;         // CTAs per cluster (1 for expand)
    int grid;            // CTAs
    size_t smem;         // dynamic shared memory bytes
};

// lora.cu
cudaError_t launch_lora(int mode, LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream,
                        LaunchInfo *info);
// Record `msg` as this thread's csgmv_last_error() and return `code`.
int set_error(int code, const char *msg);

// Whether csgmv_qkv should run as shrink + expand through a workspace.
bool qkv_split_pays(const LoraParams &p, const csgmv_batch_info &bi);
// Planes of h (parts of K) that path may write: kMaxKParts, or kDecMaxParts
// for the decode kernels.
int qkv_max_parts(const LoraParams &p, const csgmv_batch_info &bi);
// The CSGMV_PATH_* csgmv_qkv takes for p (accumulating, as csgmv_qkv) with a
// workspace of workspace_bytes (0 for none).
int qkv_path(const LoraParams &p, const csgmv_batch_info &bi, size_t workspace_bytes);
// csgmv_qkv's two-kernel paths: shrink (ps) into the fp32 workspace (a
// kWsHeader-byte header, then up to (workspace_bytes - kWsHeader) /
// (s * c * R * 4) partial-sum planes over parts of K), then the expand (pe)
// from it, on the kernels of `path` (a two-kernel CSGMV_PATH_*).
cudaError_t launch_qkv_split(LoraParams &ps, LoraParams &pe, const csgmv_batch_info &bi, cudaStream_t stream,
                             void *workspace, size_t workspace_bytes, int path);

// builder.cu
struct BuildParams {
    const int32_t *req_lens, *req_adapter;
    const int32_t *ranks_in;
    const float *scalings_in;
    int bs, num_tokens, num_loras, chunk, use_graph;
};
size_t build_smem_bytes(int bs, int max_loras);
cudaError_t launch_build(const BuildParams &p, const csgmv_batch_info &bi, cudaStream_t stream);
size_t build_lm_head_smem_bytes(int bs);
cudaError_t launch_build_lm_head(const BuildParams &p, const csgmv_batch_info &bi, cudaStream_t stream);

// embedding.cu
struct EmbeddingParams {
    const int32_t *ids;
    const uint16_t *A;      // (max_loras, R, V), or (max_loras, V, R) when transposed
    int transposed;         // 1: A is (max_loras, V, R), one contiguous row of R per id
    const uint16_t *extra;  // (max_loras, E, R) rows of extra tokens, or NULL (E = 0)
    uint16_t *out;          // (s, R)
    int64_t V, E;
    int R;
    int num_tokens, max_loras;
};
cudaError_t launch_embedding(const EmbeddingParams &p, const csgmv_batch_info &bi, cudaStream_t stream);
// out (L, V, R) = A (L, R, V) transposed per slot.
cudaError_t launch_transpose_embedding(const uint16_t *A, int64_t L, int R, int64_t V, uint16_t *out,
                                       cudaStream_t stream);
struct ExtraTokenParams {
    const int32_t *ids;
    const uint16_t *extra;  // (max_loras, E, D)
    uint16_t *out;          // (s, D), rows of extra tokens overwritten
    int64_t V, E, D;
    int num_tokens, max_loras;
};
cudaError_t launch_extra_token(const ExtraTokenParams &p, const csgmv_batch_info &bi, cudaStream_t stream);

}  // namespace csgmv
