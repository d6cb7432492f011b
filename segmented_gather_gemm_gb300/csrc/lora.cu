// Shrink, expand and fused shrink->expand kernels of the csgmv LoRA path
// (sglang chunked_backend.py run_lora_a_sgemm, run_lora_b_sgemm, run_qkv_lora,
// run_gate_up_lora; shapes from base_backend.py).
//
// Work decomposition.  The batch info groups tokens into adapter-uniform
// segments in sorted order.  A work unit is a tile of at most TM consecutive
// sorted tokens that share one slot w (consecutive segments of the same slot
// are merged up to TM tokens; longer segments are split), times one of
// `nsplit` blocks of output columns.  A thread-block cluster of CS CTAs owns a
// unit:
//   shrink  CTA q multiplies the gathered x rows of the tile by A[w] over its
//           1/CS share of K on the tensor cores (fp32 accumulators) and
//           leaves the partial h in shared memory;
//   reduce  the CS partials are summed across the cluster through
//           distributed shared memory (reduce-scatter, then all-gather), so
//           every CTA holds the full fp32 h of the tile;
//   expand  CTA q streams its 1/(nsplit*CS) share of the output columns:
//           base tile + B[w] tile in, y = base + sigma * h B^T out, with h
//           applied as bf16 hi + lo halves on the tensor cores.
// h never leaves the chip in the fused mode.  The shrink-only mode writes h
// to global memory after the reduction; the expand-only mode (cluster of 1)
// reads h from global memory instead of computing it.  The grid is persistent
// (clusters stride over units), so its size never depends on the batch and a
// captured graph stays valid for any later batch built into the same buffers.
#include <cooperative_groups.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <map>
#include <tuple>

#include "csgmv_internal.h"
#include "device_utils.cuh"

namespace cg = cooperative_groups;

namespace csgmv {
namespace {

constexpr int kThreads = 256;
constexpr int kKC = 64;        // shrink k-chunk (bf16 elements, 8 x 16-byte chunks)
constexpr int kShStages = 3;   // shrink pipeline depth
constexpr int kExStages = 3;   // expand pipeline depth

__device__ __forceinline__ void flag(int32_t *status, int bits) { atomicOr(status, bits); }

__device__ __forceinline__ int slice_of(const LoraParams &p, int col) {
    int j = 0;
    while (j + 1 < p.c && col >= p.off[j + 1]) ++j;
    return j;
}

template <int TM, int CRMAX, int MODE>
struct Tile {
    static constexpr int WM = TM / 16;              // warps along tokens
    static constexpr int WN = 8 / WM;               // warps along columns
    static constexpr int SH_TILES = (CRMAX / 8 + WN - 1) / WN;  // shrink n8 tiles per warp
    static constexpr int WCOLS = TM >= 64 ? 64 : 32;  // expand columns per warp
    static constexpr int NT = WCOLS * WN;           // expand tile width
    static constexpr int EX_TILES = WCOLS / 8;
};

template <int TM, int CRMAX, int MODE>
__device__ void process_tile(const LoraParams &p, unsigned char *smem, int q, int CS, int w, int r,
                             float sigma, int m0, int M, int nb) {
    using T = Tile<TM, CRMAX, MODE>;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp / T::WN, wn = warp % T::WN;
    int *tok = reinterpret_cast<int *>(smem + p.sm_tok);
    const int c = p.c, R = p.R;
    const int cr = c * r;
    const int crp = (cr + 7) & ~7;
    const int rp16 = (r + 15) & ~15;
    // hbf / B-tile row pitch: a power-of-two number of 16-byte chunks >= R.
    const int rpc = ((R + 15) & ~15) <= 16 ? 2 : (((R + 15) & ~15) <= 32 ? 4 : 8);
    const int rpitch = rpc * 8;
    const int rsh = pc_shift_of(rpc);

    __syncthreads();  // previous tile is done with tok[] and the stages
    for (int m = tid; m < TM; m += kThreads) {
        int t = -1;
        if (m < M) {
            t = p.permutation[m0 + m];
            if (t < 0 || t >= p.num_tokens) { flag(p.status, CSGMV_STATUS_BAD_PERMUTATION); t = -1; }
        }
        tok[m] = t;
    }
    __syncthreads();

    __nv_bfloat16 *hbf = reinterpret_cast<__nv_bfloat16 *>(smem + p.sm_hbf);
    const int hbf_half = c * TM * rpitch;  // elements of the hi (or lo) half

    if constexpr (MODE != kModeExpand) {
        // ------------------------------------------------------------------ shrink
        float *hpart = reinterpret_cast<float *>(smem + p.sm_hpart);
        const int hp = p.hrow_pitch;
        const int nkc = (int)((p.K + kKC - 1) / kKC);
        const int kc0 = (int)((int64_t)q * nkc / CS), kc1 = (int)((int64_t)(q + 1) * nkc / CS);
        const uint16_t *Aw = p.A + (int64_t)w * c * R * p.K;
        float acc[T::SH_TILES][4];
#pragma unroll
        for (int i = 0; i < T::SH_TILES; ++i)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;

        auto stage_x = [&](int st) {
            return reinterpret_cast<__nv_bfloat16 *>(smem + p.sm_stage + st * p.shrink_stage_bytes);
        };
        auto load = [&](int st, int kc) {
            __nv_bfloat16 *xs = stage_x(st);
            __nv_bfloat16 *as = xs + TM * kKC;
            const int64_t k0 = (int64_t)kc * kKC;
            for (int idx = tid; idx < TM * 8; idx += kThreads) {
                int m = idx >> 3, ch = idx & 7;
                int t = tok[m];
                int64_t kk = k0 + ch * 8;
                bool ok = t >= 0 && kk < p.K;
                const uint16_t *src = ok ? p.x + (int64_t)t * p.K + kk : p.x;
                cp_async16(xs + swz(m, ch, 8, 0), src, ok ? 16 : 0);
            }
            for (int idx = tid; idx < crp * 8; idx += kThreads) {
                int n = idx >> 3, ch = idx & 7;
                int64_t kk = k0 + ch * 8;
                bool ok = n < cr && kk < p.K;
                const uint16_t *src = ok ? Aw + (int64_t)n * p.K + kk : p.A;
                cp_async16(as + swz(n, ch, 8, 0), src, ok ? 16 : 0);
            }
        };

#pragma unroll
        for (int i = 0; i < kShStages - 1; ++i) {
            if (kc0 + i < kc1) load(i, kc0 + i);
            cp_async_commit();
        }
        for (int kc = kc0; kc < kc1; ++kc) {
            cp_async_wait<kShStages - 2>();
            __syncthreads();
            int nxt = kc + kShStages - 1;
            if (nxt < kc1) load((nxt - kc0) % kShStages, nxt);
            cp_async_commit();
            const __nv_bfloat16 *xs = stage_x((kc - kc0) % kShStages);
            const __nv_bfloat16 *as = xs + TM * kKC;
#pragma unroll
            for (int ks = 0; ks < kKC / 16; ++ks) {
                uint32_t a[4];
                ldmatrix_x4(a[0], a[1], a[2], a[3],
                            xs + swz(wm * 16 + (lane & 15), 2 * ks + (lane >> 4), 8, 0));
#pragma unroll
                for (int i = 0; i < T::SH_TILES; ++i) {
                    int j = wn + T::WN * i;
                    if (j * 8 < crp) {
                        uint32_t b0, b1;
                        ldmatrix_x2(b0, b1, as + swz(j * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1), 8, 0));
                        mma_bf16_16816(acc[i], a, b0, b1);
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // every warp is done with the stages (hpart may alias them)
#pragma unroll
        for (int i = 0; i < T::SH_TILES; ++i) {
            int j = wn + T::WN * i;
            if (j * 8 < crp) {
                int row = wm * 16 + (lane >> 2), col = j * 8 + 2 * (lane & 3);
                *reinterpret_cast<float2 *>(hpart + row * hp + col) = make_float2(acc[i][0], acc[i][1]);
                *reinterpret_cast<float2 *>(hpart + (row + 8) * hp + col) = make_float2(acc[i][2], acc[i][3]);
            }
        }

        // ------------------------------------------------------------------ reduce
        const float *hsrc_local = hpart;
        float *hred = reinterpret_cast<float *>(smem + p.sm_hred);
        const int rpr = p.rows_per_rank;
        if (CS > 1) {
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();  // partials of every CTA are written
            const int nv = crp >> 2;
            for (int idx = tid; idx < rpr * nv; idx += kThreads) {
                int rr = idx / nv, v = idx % nv;
                int row = q * rpr + rr;
                if (row >= M) continue;
                float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int peer = 0; peer < CS; ++peer) {
                    const float *rp = cluster.map_shared_rank(hpart, peer);
                    float4 v4 = *reinterpret_cast<const float4 *>(rp + row * hp + 4 * v);
                    s.x += v4.x; s.y += v4.y; s.z += v4.z; s.w += v4.w;
                }
                *reinterpret_cast<float4 *>(hred + rr * hp + 4 * v) = s;
            }
            cluster.sync();  // every CTA's rows of h are reduced
        } else {
            __syncthreads();
        }

        if constexpr (MODE == kModeShrink) {
            // Rows this CTA owns go to global h: [0, c*r) values, [c*r, c*R) zeros.
            const int row0 = CS > 1 ? q * rpr : 0;
            const int nrows = CS > 1 ? rpr : TM;
            const float *src = CS > 1 ? hred : hsrc_local;
            const int cR = c * R;
            for (int idx = tid; idx < nrows * cR; idx += kThreads) {
                int rr = idx / cR, col = idx % cR;
                int row = row0 + rr;
                if (row >= M) continue;
                int t = tok[row];
                if (t < 0) continue;
                float v = col < cr ? src[rr * hp + col] : 0.f;
                if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = v;
                else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(v);
            }
            return;
        } else {
            // All-gather the reduced rows into bf16 hi / lo halves, per slice.
            const int npair = c * TM * (rp16 >> 1);
            for (int idx = tid; idx < npair; idx += kThreads) {
                int kp = idx % (rp16 >> 1);
                int m = (idx / (rp16 >> 1)) % TM;
                int j = idx / ((rp16 >> 1) * TM);
                int k = 2 * kp;
                float v0 = 0.f, v1 = 0.f;
                if (m < M) {
                    const float *row;
                    if (CS > 1) {
                        int owner = m / rpr;
                        cg::cluster_group cluster = cg::this_cluster();
                        row = cluster.map_shared_rank(hred, owner) + (m - owner * rpr) * hp;
                    } else {
                        row = hsrc_local + m * hp;
                    }
                    if (k < r) v0 = row[j * r + k];
                    if (k + 1 < r) v1 = row[j * r + k + 1];
                }
                __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
                float l0 = v0 - __bfloat162float(h0), l1 = v1 - __bfloat162float(h1);
                int e = j * TM * rpitch + swz(m, k >> 3, rpc, rsh) + (k & 7);
                *reinterpret_cast<__nv_bfloat162 *>(hbf + e) = __halves2bfloat162(h0, h1);
                *reinterpret_cast<uint32_t *>(hbf + hbf_half + e) = pack_bf16x2(l0, l1);
            }
            __syncthreads();
        }
    } else {
        // ---------------------------------------------------------- expand input
        const int npair = c * TM * (rp16 >> 1);
        for (int idx = tid; idx < npair; idx += kThreads) {
            int kp = idx % (rp16 >> 1);
            int m = (idx / (rp16 >> 1)) % TM;
            int j = idx / ((rp16 >> 1) * TM);
            int k = 2 * kp;
            float v0 = 0.f, v1 = 0.f;
            int t = m < M ? tok[m] : -1;
            if (t >= 0) {
                int64_t base = (int64_t)t * p.ldh + j * r;
                if (p.h_f32) {
                    const float *hr = reinterpret_cast<const float *>(p.h) + base;
                    if (k < r) v0 = hr[k];
                    if (k + 1 < r) v1 = hr[k + 1];
                } else {
                    const __nv_bfloat16 *hr = reinterpret_cast<const __nv_bfloat16 *>(p.h) + base;
                    if (k < r) v0 = __bfloat162float(hr[k]);
                    if (k + 1 < r) v1 = __bfloat162float(hr[k + 1]);
                }
            }
            __nv_bfloat16 h0 = __float2bfloat16_rn(v0), h1 = __float2bfloat16_rn(v1);
            float l0 = v0 - __bfloat162float(h0), l1 = v1 - __bfloat162float(h1);
            int e = j * TM * rpitch + swz(m, k >> 3, rpc, rsh) + (k & 7);
            *reinterpret_cast<__nv_bfloat162 *>(hbf + e) = __halves2bfloat162(h0, h1);
            *reinterpret_cast<uint32_t *>(hbf + hbf_half + e) = pack_bf16x2(l0, l1);
        }
        __syncthreads();
    }

    if constexpr (MODE != kModeShrink) {
        // ------------------------------------------------------------------ expand
        const int ntot = p.off[c] - p.off[0];
        const int nparts = p.nsplit * CS;
        const int part = nb * CS + q;
        const int pcols = (((ntot + 7) >> 3) + nparts - 1) / nparts * 8;
        const int n0 = p.off[0] + part * pcols;
        const int n1 = min(p.off[c], n0 + pcols);
        if (n0 >= n1) return;
        constexpr int NT = T::NT;
        constexpr int BPC = NT / 8;  // 16-byte chunks per base-tile row
        const int ntiles = (n1 - n0 + NT - 1) / NT;
        const int bchunks = rp16 >> 3;
        const uint16_t *Bw = p.B + (int64_t)w * p.N * R;
        const int ksteps = rp16 >> 4;

        auto stage_b = [&](int st) {
            return reinterpret_cast<__nv_bfloat16 *>(smem + p.sm_ex + st * p.ex_stage_bytes);
        };
        auto load = [&](int st, int it) {
            __nv_bfloat16 *bs = stage_b(st);
            __nv_bfloat16 *bt = bs + TM * NT;
            const int nt0 = n0 + it * NT;
            if (p.accumulate) {
                for (int idx = tid; idx < M * BPC; idx += kThreads) {
                    int m = idx / BPC, ch = idx % BPC;
                    int col = nt0 + ch * 8;
                    int t = tok[m];
                    if (t >= 0 && col < n1)
                        cp_async16(bs + swz(m, ch, BPC, 0), p.y + (int64_t)t * p.N + col, 16);
                }
            }
            for (int idx = tid; idx < NT * bchunks; idx += kThreads) {
                int n = idx / bchunks, ch = idx % bchunks;
                int col = nt0 + n;
                int kk = ch * 8;
                int bytes = col < n1 ? min(16, max(0, (r - kk) * 2)) : 0;
                const uint16_t *src = bytes ? Bw + (int64_t)col * R + kk : p.B;
                cp_async16(bt + swz(n, ch, rpc, rsh), src, bytes);
            }
        };

#pragma unroll
        for (int i = 0; i < kExStages - 1; ++i) {
            if (i < ntiles) load(i, i);
            cp_async_commit();
        }
        for (int it = 0; it < ntiles; ++it) {
            cp_async_wait<kExStages - 2>();
            __syncthreads();
            if (it + kExStages - 1 < ntiles) load((it + kExStages - 1) % kExStages, it + kExStages - 1);
            cp_async_commit();
            __nv_bfloat16 *bs = stage_b(it % kExStages);
            const __nv_bfloat16 *bt = bs + TM * NT;
            const int nt0 = n0 + it * NT;

            float acc[T::EX_TILES][4];
#pragma unroll
            for (int i = 0; i < T::EX_TILES; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[i][e] = 0.f;
            for (int ks = 0; ks < ksteps; ++ks) {
                int cur = -1;
                uint32_t ahi[4], alo[4];
#pragma unroll
                for (int i = 0; i < T::EX_TILES; ++i) {
                    int lc = wn * T::WCOLS + 8 * i;
                    int col8 = nt0 + lc;
                    if (col8 >= n1) continue;
                    int j = slice_of(p, col8);
                    if (j != cur) {
                        const __nv_bfloat16 *hs = hbf + j * TM * rpitch;
                        int e = swz(wm * 16 + (lane & 15), 2 * ks + (lane >> 4), rpc, rsh);
                        ldmatrix_x4(ahi[0], ahi[1], ahi[2], ahi[3], hs + e);
                        ldmatrix_x4(alo[0], alo[1], alo[2], alo[3], hs + hbf_half + e);
                        cur = j;
                    }
                    uint32_t b0, b1;
                    ldmatrix_x2(b0, b1, bt + swz(lc + (lane & 7), 2 * ks + ((lane >> 3) & 1), rpc, rsh));
                    mma_bf16_16816(acc[i], ahi, b0, b1);
                    mma_bf16_16816(acc[i], alo, b0, b1);
                }
            }
            // y = base + sigma * acc, written back into the base tile.
#pragma unroll
            for (int i = 0; i < T::EX_TILES; ++i) {
                int lc = wn * T::WCOLS + 8 * i + 2 * (lane & 3);
                if (nt0 + wn * T::WCOLS + 8 * i >= n1) continue;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    int row = wm * 16 + (lane >> 2) + 8 * hh;
                    if (row >= M) continue;
                    uint32_t *ptr = reinterpret_cast<uint32_t *>(bs + swz(row, lc >> 3, BPC, 0) + (lc & 7));
                    float2 b = p.accumulate ? unpack_bf16x2(*ptr) : make_float2(0.f, 0.f);
                    *ptr = pack_bf16x2(b.x + sigma * acc[i][2 * hh], b.y + sigma * acc[i][2 * hh + 1]);
                }
            }
            __syncthreads();
            for (int idx = tid; idx < M * BPC; idx += kThreads) {
                int m = idx / BPC, ch = idx % BPC;
                int col = nt0 + ch * 8;
                int t = tok[m];
                if (t >= 0 && col < n1)
                    *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + col) =
                        *reinterpret_cast<const uint4 *>(bs + swz(m, ch, BPC, 0));
            }
        }
        cp_async_wait<0>();
    }
}

// Rows of a unit whose slot has rank 0: the shrink writes zero h rows, the
// non-accumulating expand writes zero outputs; otherwise nothing is touched.
template <int TM, int MODE>
__device__ void zero_rows(const LoraParams &p, int q, int CS, int p0, int p1, int nb) {
    const int tid = threadIdx.x;
    if constexpr (MODE == kModeShrink) {
        const int cR = p.c * p.R;
        // CTA q of the cluster clears rows q, q + CS, ...
        for (int m = p0 + q; m < p1; m += CS) {
            int t = p.permutation[m];
            if (t < 0 || t >= p.num_tokens) continue;
            for (int col = tid; col < cR; col += kThreads) {
                if (p.h_f32) reinterpret_cast<float *>(p.h)[(int64_t)t * p.ldh + col] = 0.f;
                else reinterpret_cast<__nv_bfloat16 *>(p.h)[(int64_t)t * p.ldh + col] = __float2bfloat16_rn(0.f);
            }
        }
    } else if constexpr (MODE == kModeExpand) {
        if (p.accumulate) return;
        const int ntot = p.off[p.c] - p.off[0];
        const int nparts = p.nsplit * CS;
        const int part = nb * CS + q;
        const int pcols = (((ntot + 7) >> 3) + nparts - 1) / nparts * 8;
        const int n0 = p.off[0] + part * pcols;
        const int n1 = min(p.off[p.c], n0 + pcols);
        const int nch = (n1 - n0 + 7) >> 3;
        if (nch <= 0) return;
        for (int m = p0; m < p1; ++m) {
            int t = p.permutation[m];
            if (t < 0 || t >= p.num_tokens) continue;
            for (int ch = tid; ch < nch; ch += kThreads)
                *reinterpret_cast<uint4 *>(p.y + (int64_t)t * p.N + n0 + 8 * ch) = make_uint4(0, 0, 0, 0);
        }
    }
}

template <int TM, int CRMAX, int MODE>
__device__ void process_run(const LoraParams &p, unsigned char *smem, int q, int CS, int w, int p0,
                            int p1, int nb) {
    p0 = max(p0, 0);
    p1 = min(p1, p.num_tokens);  // sorted positions never exceed the token count
    if (p0 >= p1) return;
    if (w < 0 || w >= p.max_loras) {
        if (q == 0 && threadIdx.x == 0) flag(p.status, CSGMV_STATUS_BAD_ADAPTER);
        return;
    }
    const int r = p.lora_ranks[w];
    if (r < 0 || r > p.R) {
        if (q == 0 && threadIdx.x == 0) flag(p.status, CSGMV_STATUS_BAD_RANK);
        return;
    }
    if (r == 0) {
        zero_rows<TM, MODE>(p, q, CS, p0, p1, nb);
        return;
    }
    const float sigma = p.scalings[w];
    for (int m0 = p0; m0 < p1; m0 += TM)
        process_tile<TM, CRMAX, MODE>(p, smem, q, CS, w, r, sigma, m0, min(TM, p1 - m0), nb);
}

template <int TM, int CRMAX, int MODE>
__global__ void __launch_bounds__(kThreads, TM <= 32 ? 2 : 1) lora_kernel(const __grid_constant__ LoraParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    int CS = 1, q = 0;
    if constexpr (MODE != kModeExpand) {
        cg::cluster_group cluster = cg::this_cluster();
        CS = (int)cluster.num_blocks();
        q = (int)cluster.block_rank();
    }
    const int cid = blockIdx.x / CS, ncl = gridDim.x / CS;

    const int nseg = *p.num_segments_dev;
    const int chunk = max(1, *p.max_len_dev);
    const int G = chunk >= TM ? 1 : TM / chunk;          // segments merged per unit
    const int SUB = chunk > TM ? (chunk + TM - 1) / TM : 1;  // token tiles per segment
    const int ngroups = (nseg + G - 1) / G;
    const int64_t nunits = (int64_t)ngroups * SUB * p.nsplit;

    for (int64_t u = cid; u < nunits; u += ncl) {
        const int nb = (int)(u % p.nsplit);
        const int64_t rest = u / p.nsplit;
        const int sub = (int)(rest % SUB);
        const int grp = (int)(rest / SUB);
        const int s0 = grp * G, s1 = min(nseg, s0 + G);
        if (G == 1) {
            const int pb = p.seg_indptr[s0], pe = p.seg_indptr[s0 + 1];
            const int p0 = pb + sub * TM;
            const int p1 = (sub == SUB - 1) ? pe : min(pe, p0 + TM);
            if (p0 < p1) process_run<TM, CRMAX, MODE>(p, smem, q, CS, p.weight_indices[s0], p0, p1, nb);
        } else {
            int k = s0;
            while (k < s1) {
                const int w = p.weight_indices[k];
                int e = k + 1;
                while (e < s1 && p.weight_indices[e] == w) ++e;
                const int p0 = p.seg_indptr[k], p1 = p.seg_indptr[e];
                if (p0 < p1) process_run<TM, CRMAX, MODE>(p, smem, q, CS, w, p0, p1, nb);
                k = e;
            }
        }
    }
    if constexpr (MODE != kModeExpand) {
        if (CS > 1) cg::this_cluster().sync();  // peers may still read this CTA's shared memory
    }
}

// ----------------------------------------------------------------------------- host side

using KernelFn = void (*)(LoraParams);

template <int TM, int CRMAX, int MODE>
KernelFn kernel_ptr() { return lora_kernel<TM, CRMAX, MODE>; }

KernelFn pick_kernel(int mode, int tm, int crmax) {
#define CSGMV_PICK(TM_, CR_)                                                     \
    if (tm == TM_ && crmax == CR_) {                                             \
        if (mode == kModeFused) return kernel_ptr<TM_, CR_, kModeFused>();       \
        if (mode == kModeShrink) return kernel_ptr<TM_, CR_, kModeShrink>();     \
    }
    CSGMV_PICK(16, 64)
    CSGMV_PICK(16, 192)
    CSGMV_PICK(64, 192)
    CSGMV_PICK(128, 64)
    CSGMV_PICK(128, 128)
#undef CSGMV_PICK
    if (mode == kModeExpand) {
        if (tm == 16) return kernel_ptr<16, 8, kModeExpand>();
        if (tm == 64) return kernel_ptr<64, 8, kModeExpand>();
        if (tm == 128) return kernel_ptr<128, 8, kModeExpand>();
    }
    return nullptr;
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

struct OccKey {
    KernelFn fn;
    int cluster;
    size_t smem;
    int dev;
    bool operator<(const OccKey &o) const {
        return std::tie(fn, cluster, smem, dev) < std::tie(o.fn, o.cluster, o.smem, o.dev);
    }
};

std::mutex g_mu;
std::map<OccKey, int> g_occ;          // co-resident clusters (or CTAs) per launch shape
std::map<std::pair<KernelFn, int>, bool> g_attr;

cudaError_t ensure_attrs(KernelFn fn, int dev, int cluster) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(fn, dev);
    if (g_attr.count(key)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    g_attr[key] = true;
    return cudaSuccess;
}

cudaError_t resident_units(KernelFn fn, int dev, int cluster, size_t smem, int *out) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find({fn, cluster, smem, dev});
        if (it != g_occ.end()) { *out = it->second; return cudaSuccess; }
    }
    int n = 0;
    cudaError_t e;
    if (cluster > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
    } else {
        int per_sm = 0, sms = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = per_sm * sms;
    }
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[{fn, cluster, smem, dev}] = n;
    *out = n;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_lora(int mode, LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream,
                        LaunchInfo *info) {
    const int cR = p.c * p.R;
    const int s = p.num_tokens;
    // Token tile: small tiles for decode-like batches (few tokens per slot),
    // 128-token tiles (64 when c*R > 128) for prefill.
    const int slots_used = std::max(1, std::min(bi.num_loras > 0 ? bi.num_loras : bi.max_loras,
                                                std::max(1, bi.bs)));
    const bool small = s <= 64 * slots_used || s <= 1024;
    int tm, crmax;
    if (mode == kModeExpand) {
        tm = small ? 16 : 128;
        crmax = 8;
    } else {
        crmax = cR <= 64 ? 64 : (cR <= 128 ? 128 : 192);
        if (small) { tm = 16; if (crmax == 128) crmax = 192; }
        else { tm = crmax == 192 ? 64 : 128; }
        if (tm == 16 && crmax == 64) crmax = 64;
    }
    const int cluster = mode == kModeExpand ? 1 : 8;
    KernelFn fn = pick_kernel(mode, tm, crmax);
    if (!fn) return cudaErrorInvalidValue;

    // Shared memory carve-up.
    const int wn = 8 / (tm / 16);
    const int wcols = tm >= 64 ? 64 : 32;
    const int nt = wcols * wn;
    const int rp = round_up(std::max(p.R, 1), 16);
    const int rpc = rp <= 16 ? 2 : (rp <= 32 ? 4 : 8);
    const int rpitch = rpc * 8;
    p.hrow_pitch = crmax + 4;
    p.rows_per_rank = cluster > 1 ? tm / cluster : tm;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 127) / 128 * 128; return (int)o; };
    p.sm_tok = take((size_t)tm * 4);
    p.shrink_stage_bytes = mode == kModeExpand ? 0 : (tm * kKC + crmax * kKC) * 2;
    p.ex_stage_bytes = mode == kModeShrink ? 0 : (tm * nt + nt * rpitch) * 2;
    const size_t shrink_bytes = (size_t)kShStages * p.shrink_stage_bytes;
    const size_t hpart_bytes = mode == kModeExpand ? 0 : (size_t)tm * p.hrow_pitch * 4;
    const size_t hred_bytes = (mode == kModeExpand || cluster == 1) ? 0 : (size_t)p.rows_per_rank * p.hrow_pitch * 4;
    const size_t hbf_bytes = mode == kModeShrink ? 0 : (size_t)2 * p.c * tm * rpitch * 2;
    const size_t ex_bytes = (size_t)kExStages * p.ex_stage_bytes;
    const size_t budget = 227 * 1024;
    const size_t plain = 128 * 5 + (size_t)tm * 4 + shrink_bytes + hpart_bytes + hred_bytes + hbf_bytes + ex_bytes;
    if (plain <= budget) {
        p.sm_stage = take(shrink_bytes);
        p.sm_hpart = take(hpart_bytes);
        p.sm_hred = take(hred_bytes);
        p.sm_hbf = take(hbf_bytes);
        p.sm_ex = take(ex_bytes);
        p.ex_prefetch = 1;
    } else {
        // The shrink stages, the fp32 partials and the expand stages are live
        // one after the other, so they share one region.
        p.sm_stage = take(std::max(shrink_bytes, std::max(hpart_bytes, ex_bytes)));
        p.sm_hpart = p.sm_stage;
        p.sm_ex = p.sm_stage;
        p.sm_hred = take(hred_bytes);
        p.sm_hbf = take(hbf_bytes);
        p.ex_prefetch = 0;
    }
    const size_t smem = off;
    if (smem > budget) return cudaErrorInvalidConfiguration;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = ensure_attrs(fn, dev, cluster);
    if (e != cudaSuccess) return e;
    int resident = 0;
    e = resident_units(fn, dev, cluster, smem, &resident);
    if (e != cudaSuccess) return e;

    // Upper bound on token tiles of any batch these buffers can hold.
    const int chunk = std::max(1, bi.chunk_size);
    const int tiles_ub = (s + tm - 1) / tm + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    if (mode == kModeShrink) {
        p.nsplit = 1;
    } else {
        // Split the output columns further when the tiles alone cannot fill
        // the co-resident clusters.
        const int ntot = p.off[p.c] - p.off[0];
        const int max_split = std::max(1, ntot / (cluster * nt));
        int want = (resident + tiles_ub - 1) / std::max(tiles_ub, 1);
        p.nsplit = std::max(1, std::min(want, max_split));
    }
    (void)chunk;
    const int64_t units_ub = (int64_t)tiles_ub * p.nsplit;
    const int nclusters = (int)std::max<int64_t>(1, std::min<int64_t>(resident, units_ub));

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nclusters * cluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (info) {
        info->tm = tm;
        info->crmax = crmax;
        info->cluster = cluster;
        info->grid = nclusters * cluster;
        info->smem = smem;
    }
    e = cudaLaunchKernelEx(&cfg, fn, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csgmv
