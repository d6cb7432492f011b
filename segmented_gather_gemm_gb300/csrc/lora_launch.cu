// Host side of the LoRA kernels: tile / cluster / pipeline choice, shared
// memory carve-up, TMA descriptors, cluster launch.
#include <cudaTypedefs.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "lora_decode.cuh"
#include "lora_small.cuh"
#include "lora_wide.cuh"
#include "lora_stream.cuh"

namespace csgmv {

const void *lora_kernel_fused(int tm, int rmax, bool tc);
const void *lora_kernel_shrink(int tm, int rmax, bool tc);
const void *lora_kernel_expand(int tm, int rmax, bool tc);
const void *lora_kernel_small(int mode, int tm, int rmax);
const void *lora_kernel_stream();
const void *lora_kernel_sshrink();
const void *lora_kernel_decode(int which, int rmax);
const void *lora_kernel_wide(int tm, int rmax);

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_mu;
std::map<std::pair<const void *, int>, bool> g_attr;                     // (kernel, device) attributes set
std::map<std::tuple<const void *, int, size_t, int>, int> g_occupancy;  // (kernel, cluster, smem, dev)

cudaError_t encoder() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_encode) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// 2D bf16 tensor map: `inner` elements per row (contiguous), `outer` rows of
// `row_bytes` bytes, box of box_inner x box_outer elements.
bool encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
    if (!g_encode) return false;  // every launcher resolves it (encoder()) first
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3D bf16 view of a row-major (outer, inner) tensor as (64-column chunks,
// rows, chunk index): dims {64, outer, inner / 64}, strides {row_bytes, 128},
// box {64, box_rows, box_chunks}, 128-byte swizzle.  One load then fills
// box_chunks tiles of box_rows x 64, one after the other.
bool encode_3d_chunks(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_rows, uint32_t box_chunks) {
    if (!g_encode || inner % 64 != 0 || box_rows > 256 || box_chunks > 256) return false;
    cuuint64_t dims[3] = {64, outer, inner / 64};
    cuuint64_t strides[2] = {row_bytes, 128};
    cuuint32_t box[3] = {64, box_rows, box_chunks};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

CUtensorMapSwizzle swizzle_for_row_bytes(int bytes) {
    return bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
         : bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
         : bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
}

// B of the expand: one (L, N, R) tensor in tmB (box R x box_rows), or, with
// separate slice tensors, slice j in tmBs[j] (box R x 64); unused maps are
// copies of a valid one.
bool encode_b_maps(CUtensorMap *tmB, CUtensorMap *tmBs, const LoraParams &p, int L, uint32_t box_rows) {
    const CUtensorMapSwizzle sw = swizzle_for_row_bytes(p.R * 2);
    if (!p.b_tuple) {
        if (!encode_2d(tmB, p.B, (uint64_t)p.R, (uint64_t)L * p.N, (uint64_t)p.R * 2, p.R, box_rows, sw))
            return false;
        for (int j = 0; j < kMaxSlices; ++j) tmBs[j] = *tmB;
        return true;
    }
    for (int j = 0; j < kMaxSlices; ++j) {
        const int jj = j < p.c ? j : 0;
        if (!encode_2d(&tmBs[j], p.Bs[jj], (uint64_t)p.R, (uint64_t)L * p.b_rows[jj], (uint64_t)p.R * 2, p.R, 64,
                       sw))
            return false;
    }
    *tmB = tmBs[0];
    return true;
}
bool encode_b(TmaKernelParams &k, int L, uint32_t box_rows) { return encode_b_maps(&k.tmB, k.tmBs, k.p, L, box_rows); }

cudaError_t ensure_attrs(const void *fn, int dev, int cluster) {
    std::lock_guard<std::mutex> lk(g_mu);
    auto key = std::make_pair(fn, dev);
    if (g_attr.count(key)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    // the whole unified L1 as shared memory: an SM configured for one kernel
    // then also takes the CTAs of a dependent kernel launched behind it
    // without first draining to change its carve-out
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    (void)cluster;  // clusters of up to 16 CTAs
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    g_attr[key] = true;
    return cudaSuccess;
}

// Programmatic dependent launch: the kernel's CTAs may launch and set up
// their barriers while the kernel before it in the stream (typically the
// batch-info builder, which allows it at its start) is still running; every
// LoRA kernel waits for that kernel on the device before reading global memory.
void set_dependent_launch(cudaLaunchAttribute *a) {
    a->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a->val.programmaticStreamSerializationAllowed = 1;
}

// Co-resident clusters of `cluster` CTAs (or CTAs when cluster == 1).
cudaError_t resident(const void *fn, int dev, int cluster, size_t smem, int *out, int threads = kTmaThreads) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occupancy.find({fn, cluster, smem, dev});
        if (it != g_occupancy.end()) { *out = it->second; return cudaSuccess; }
    }
    int n = 0;
    cudaError_t e;
    if (cluster > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
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
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = per_sm * sms;
    }
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occupancy[{fn, cluster, smem, dev}] = n;
    *out = n;
    return cudaSuccess;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    TmaKernelParams *k;
    size_t bytes;
};

// Shared-memory carve-up for the given ring depths; returns the bytes needed.
// The fp32 partials of the shrink alias the shrink ring: they are written
// after the last chunk of a unit is consumed and read by the cluster before
// any copy of the next unit lands there.
size_t carve(TmaKernelParams &k, int mode, int tm, int cs, int S1, int S2, bool tc) {
    const int nb64 = tc ? kTcCols / 64 : (tm >= 128 ? 1 : (tm >= 64 ? 2 : 4));
    const int nt = 64 * nb64;
    const int R = k.p.R;
    const int cR = k.p.c * R;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = align_up(off, align);
        size_t o = off;
        off += bytes;
        return (int)o;
    };
    k.S1 = mode == kModeExpand ? 1 : S1;
    k.S2 = mode == kModeShrink ? 1 : S2;
    k.hp = align_up((size_t)cR, 8) + 4;
    k.a_rows = (int)align_up((size_t)cR, 16);
    k.o_bar = take((size_t)(2 * k.S1 + 2 * k.S2) * 8, 8);
    k.o_tc = tc ? take(64, 16) : 0;
    const size_t ah_bytes = tc ? (size_t)k.ah_slices * 2 * kTcAhBytes : 0;
    k.o_run = take((size_t)(5 * k.runcap + 1 + 32) * 4, 16);
    k.o_tok = take((size_t)tm * 4, 16);
    if (mode != kModeExpand) {
        k.sh_a = tm * 128;
        k.sh_stage = (int)align_up((size_t)tm * 128 + (size_t)k.a_rows * 128, 1024);
        // the tensor-core expand's h operand tiles alias the ring as well:
        // they are written after the reduction, when the ring is idle
        const size_t ring = std::max({(size_t)k.S1 * k.sh_stage, (size_t)tm * k.hp * 4, ah_bytes});
        k.o_sh = take(ring, 1024);
        k.o_hpart = k.o_sh;
        k.o_ah = k.o_sh;
        k.o_hred = cs > 1 ? take((size_t)(tm / cs) * k.hp * 4, 16) : k.o_hpart;
    } else {
        k.sh_a = 0;
        k.sh_stage = 0;
        k.o_sh = k.o_hpart = k.o_hred = 0;
        k.o_ah = tc ? take(ah_bytes, 1024) : 0;
    }
    if (mode != kModeShrink) {
        k.ex_b = nb64 * tm * 128;
        k.ex_stage = (int)align_up((size_t)k.ex_b + (size_t)nt * 2 * R, 1024);
        k.o_ex = take((size_t)k.S2 * k.ex_stage, 1024);
    } else {
        k.ex_b = k.ex_stage = k.o_ex = 0;
    }
    return off + 1024;  // slack for aligning the dynamic window to 1024 bytes
}


// Most slices that one CTA's column range spans, for nsplit * cs column
// parts (the device split in column_range()).
int max_slice_span(const LoraParams &p, int parts) {
    const int ntot = p.off[p.c] - p.off[0];
    const int nblk = (ntot + 63) / 64;
    auto slice_of = [&](int col) {
        int j = 0;
        while (j + 1 < p.c && col >= p.off[j + 1]) ++j;
        return j;
    };
    int span = 1;
    for (int part = 0; part < parts; ++part) {
        const int b0 = (int)((int64_t)part * nblk / parts), b1 = (int)((int64_t)(part + 1) * nblk / parts);
        const int n0 = p.off[0] + 64 * b0, n1 = std::min(p.off[p.c], p.off[0] + 64 * b1);
        if (n1 > n0) span = std::max(span, slice_of(n1 - 1) - slice_of(n0) + 1);
    }
    return span;
}

// Shared-memory carve-up of the small-tile kernel.
// Columns per expand stage of the small-tile kernel (SmallGeo::NT).
int small_stage_cols(int mode, int tm) { return tm == 16 && mode == kModeExpand ? 512 : 256; }

size_t carve_small(TmaKernelParams &k, int mode, int tm, int cs, int S2) {
    const int R = k.p.R;
    const int cR = k.p.c * R;
    const int nkc = (int)((k.p.K + 63) / 64);
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = align_up(off, align);
        size_t o = off;
        off += bytes;
        return (int)o;
    };
    k.S1 = 1;
    k.S2 = mode == kModeShrink ? 1 : S2;
    k.hp = (int)align_up((size_t)cR, 8) + 4;
    k.a_rows = (int)align_up((size_t)cR, 16);
    k.o_bar = take((size_t)(1 + 2 * k.S2) * 8, 8);
    k.o_run = take((size_t)(5 * k.runcap + 1 + 32) * 4, 16);
    k.o_tok = take((size_t)tm * 4, 16);
    k.kc_per = 0;
    k.xpitch = 16;
    k.o_sh = k.o_ah = k.o_hred = 0;
    // h partials (shrink) and, right after them, the per-warp epilogue scratch
    // tiles (expand): 16 rows x (NT / WN) columns each, rows padded by 16 bytes
    const int nt = small_stage_cols(mode, tm);
    const int wcols = nt / (kConsumerWarps / (tm / 16));
    k.o_hpart = take((size_t)tm * k.hp * 4 + (size_t)kConsumerWarps * 16 * (wcols * 2 + 16), 16);
    k.wscr_off = (int)align_up((size_t)tm * k.hp * 4, 16);
    if (mode != kModeExpand) {
        k.kc_per = (nkc + cs - 1) / cs;
        k.xpitch = k.kc_per * 128 + 16;  // 16 bytes of padding: conflict-free ldmatrix rows
        k.o_sh = take((size_t)tm * k.xpitch, 16);
        k.o_ah = take((size_t)k.kc_per * k.a_rows * 128, 1024);
        k.o_hred = cs > 1 ? take((size_t)tm * k.hp * 4, 16) : k.o_hpart;  // every CTA's full h
    }
    k.ypitch = 16;
    k.ex_b = k.ex_stage = k.o_ex = 0;
    if (mode != kModeShrink) {
        k.ypitch = nt * 2 + 16;
        k.ex_b = (int)align_up((size_t)tm * k.ypitch, 1024);
        k.ex_stage = (int)align_up((size_t)k.ex_b + (size_t)nt * R * 2, 1024);
        k.o_ex = take((size_t)k.S2 * k.ex_stage, 1024);
    }
    return off + 1024;  // slack for aligning the dynamic window to 1024 bytes
}

}  // namespace

// 16- and 32-token tiles (decode) on the small-tile kernel.  Returns
// cudaErrorInvalidConfiguration when no cluster shape fits; the caller then
// takes the streaming kernel.
cudaError_t launch_lora_small(int mode, LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream,
                              LaunchInfo *info, int rmax, int tm) {
    const void *fn = lora_kernel_small(mode, tm, rmax);
    if (!fn) return cudaErrorInvalidConfiguration;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    TmaKernelParams k;
    memset(&k, 0, sizeof k);
    k.p = p;
    k.max_segments = bi.max_segments;
    k.runcap = std::max(1, std::min(bi.max_segments, bi.max_loras + std::max(bi.max_bs, 1)));
    const size_t budget = 227 * 1024;
    const int s = p.num_tokens;
    const int slots = std::max(1, std::min(std::max(bi.bs, 1), bi.num_loras > 0 ? bi.num_loras : bi.max_loras));
    // expected tiles: full tiles plus about half a partial tile per slot run
    const int tiles_est = std::max(slots, s / tm + slots / 2);
    const int ncols = p.off[p.c] - p.off[0];
    // Cluster size: the fewest waves of units, then the largest cluster (the
    // finest split of each unit's work).
    const int cs_list[5] = {16, 8, 4, 2, 1};
    int best_waves = 1 << 30, best_cs = 0, best_res = 0, best_S2 = 2;
    for (int ci = 0; ci < 5; ++ci) {
        const int cs = mode == kModeExpand ? 1 : cs_list[ci];
        if (mode == kModeExpand && ci > 0) break;
        if (tm % cs) continue;
        const int nt = small_stage_cols(mode, tm);
        const int stages = std::max(1, (ncols / cs + nt - 1) / nt);
        int S2 = std::min(8, std::max(2, stages + 1));
        size_t smem = carve_small(k, mode, tm, cs, S2);
        while (smem > budget && S2 > 2) smem = carve_small(k, mode, tm, cs, --S2);
        if (smem > budget) continue;
        if (ensure_attrs(fn, dev, cs) != cudaSuccess) continue;
        int res = 0;
        if (resident(fn, dev, cs, smem, &res) != cudaSuccess || res < 1) continue;
        const int waves = (tiles_est + res - 1) / res;
        if (waves < best_waves) { best_waves = waves; best_cs = cs; best_res = res; best_S2 = S2; }
    }
    if (best_cs == 0) return cudaErrorInvalidConfiguration;
    const int cs = best_cs;
    const size_t smem = carve_small(k, mode, tm, cs, best_S2);

    const int tiles_ub = (s + tm - 1) / tm + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    if (mode == kModeShrink) {
        k.p.nsplit = 1;
    } else {
        // column blocks per tile: enough units for every resident cluster
        // (counted from the expected tiles), each block at least 4 x 64 columns
        const int nblk = (ncols + 63) / 64;
        const int max_split = std::max(1, nblk / (cs * 4));
        k.p.nsplit = std::max(1, std::min(best_res / std::max(tiles_est, 1), max_split));
    }
    const int64_t units_ub = (int64_t)tiles_ub * k.p.nsplit;
    const int nclusters = (int)std::max<int64_t>(1, std::min<int64_t>(best_res, units_ub));

    const int L = bi.max_loras;
    const int cR = p.c * p.R;
    bool ok = true;
    if (mode != kModeExpand)
        ok = ok && encode_2d(&k.tmA, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 64, k.a_rows,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (mode != kModeShrink)
        ok = ok && encode_b(k, L, 256);
    if (mode == kModeExpand) k.tmA = k.tmB;
    if (mode == kModeShrink) k.tmB = k.tmA;
    k.tmX = k.tmY = k.tmXg = k.tmA;
    if (!ok) return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nclusters * cs, 1, 1);
    cfg.blockDim = dim3(kConsumerThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_dependent_launch(&attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (info) {
        info->tm = tm;
        info->crmax = rmax;
        info->cluster = cs;
        info->grid = nclusters * cs;
        info->smem = smem;
    }
    void *args[1] = {&k};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Shared-memory carve-up of the streaming expand kernel for ring depth S;
// returns the bytes needed (with slack for aligning the window to 1024).
size_t carve_stream(StreamParams &k, int Sy) {
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = align_up(off, align);
        size_t o = off;
        off += bytes;
        return (int)o;
    };
    k.Sy = Sy;
    k.Sb = kStBSlots;
    k.y_slot_bytes = kStBoxes * kStTileBytes;
    k.b_slot_bytes = kStCols * k.p.R * 2;
    k.o_bar = take((size_t)(3 * k.Sb + 2 * Sy + 2 * kStAcc + 4) * 8 + 16 + (size_t)k.Sb * 4, 16);
    k.o_run = take((size_t)(8 * k.runcap + 1 + 32) * 4, 16);  // run table cut at token gaps
    k.o_tok = take((size_t)(2 * 128 + 8) * 4, 16);
    k.o_bring = take((size_t)k.Sb * k.b_slot_bytes, 1024);
    k.o_yring = take((size_t)Sy * k.y_slot_bytes, 1024);
    // at least 116 KB, so that one CTA holds an SM (and its 512 TMEM columns)
    return std::max(off + 1024, (size_t)116 * 1024);
}

// Shared-memory carve-up of the streaming shrink kernel for ring depth S.
size_t carve_sshrink(ShrinkParams &k, int S) {
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = align_up(off, align);
        size_t o = off;
        off += bytes;
        return (int)o;
    };
    k.S = S;
    k.a_off = k.chunks * 128 * 128;
    k.a_bytes = (int)(align_up((size_t)k.p.c * k.p.R, 16) * 128);
    k.stage_bytes = (int)align_up((size_t)k.a_off + (size_t)k.chunks * k.a_bytes, 1024);
    k.o_bar = take((size_t)(2 * S + 6) * 8 + 16, 16);
    k.o_run = take((size_t)(8 * k.runcap + 1 + 32) * 4, 16);  // run table cut at token gaps
    k.o_tok = take((size_t)(2 * 128 + 2) * 4, 16);
    k.o_ring = take((size_t)S * k.stage_bytes, 1024);
    return std::max(off + 1024, (size_t)116 * 1024);
}

// Shrink on 128-token tiles: the streaming tcgen05 kernel, one CTA per SM.
// K may be cut into up to max_parts parts (more than one only into an fp32
// workspace of max_parts planes of p.h_plane elements); the kernel picks the
// count from the exact tile count and writes it to *parts_dev (device) when
// that is not NULL.
cudaError_t launch_lora_sshrink(LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream, LaunchInfo *info,
                                int max_parts, int *parts_dev) {
    const void *fn = lora_kernel_sshrink();
    cudaError_t e = encoder();  // the tensor-map encoder, resolved on first use
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    ShrinkParams k;
    memset(&k, 0, sizeof k);
    k.p = p;
    k.max_segments = bi.max_segments;
    k.runcap = std::max(1, std::min(bi.max_segments, bi.max_loras + std::max(bi.max_bs, 1)));
    const size_t budget = 227 * 1024;
    // the most K chunks per stage that still leave three stages, else two
    // chunks and as many stages as fit (up to eight)
    int S = 8;
    size_t smem = 0;
    for (k.chunks = kShChunksMax; k.chunks >= 2; --k.chunks) {
        S = 8;
        smem = carve_sshrink(k, S);
        while (smem > budget && S > 2) smem = carve_sshrink(k, --S);
        if (smem <= budget && (S >= 3 || k.chunks == 2)) break;
    }
    if (smem > budget) return cudaErrorInvalidConfiguration;
    e = ensure_attrs(fn, dev, 1);
    if (e != cudaSuccess) return e;
    int res = 0;
    e = resident(fn, dev, 1, smem, &res, kShThreads);
    if (e != cudaSuccess) return e;
    if (res < 1) return cudaErrorInvalidConfiguration;

    const int s = p.num_tokens;
    // tiles: one per 128 tokens, plus a partial one per slot run and per request
    const int tiles_ub = (s + 127) / 128 + std::max(bi.bs, 1) + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    k.max_parts = std::max(1, max_parts);
    k.parts_out = parts_dev;
    k.plane = p.h_plane;
    const int64_t units_ub = (int64_t)tiles_ub * k.max_parts;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(res, units_ub));

    const int L = bi.max_loras;
    const int cR = p.c * p.R;
    bool ok = encode_2d(&k.tmX, p.x, (uint64_t)p.K, (uint64_t)s, (uint64_t)p.K * 2, 64, 128,
                        CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmXg, p.x, (uint64_t)p.K, (uint64_t)s, (uint64_t)p.K * 2, 64, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    for (int i = 0; i < 4; ++i)
        ok = ok && encode_2d(&k.tmXp[i], p.x, (uint64_t)p.K, (uint64_t)s, (uint64_t)p.K * 2, 64, 64u >> i,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmA, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 64, 16,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmA32, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 64, 32,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmA64, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;
    // one-instruction stages when K splits into whole chunks (else the 2-D maps)
    k.use3d = p.K % 64 == 0 &&
              encode_3d_chunks(&k.tmX3, p.x, (uint64_t)p.K, (uint64_t)s, (uint64_t)p.K * 2, 128, k.chunks) &&
              encode_3d_chunks(&k.tmA3, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2,
                               (uint32_t)k.a_bytes / 128, k.chunks);
    for (int l = 0; l < 3 && k.use3d; ++l)
        k.use3d = encode_3d_chunks(&k.tmA3s[l], p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 16u << l,
                                   k.chunks);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kShThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_dependent_launch(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (info) {
        info->tm = 128;
        info->crmax = p.R;
        info->cluster = 1;
        info->grid = grid;
        info->smem = smem;
    }
    void *args[1] = {&k};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Expand-only calls on 128-token tiles: the streaming tcgen05 kernel, one CTA
// per SM.  Units are (tile, column block inside one slice); the column block
// is sized so that every CTA gets about sixteen units, and holds at least
// 16 R columns.
cudaError_t launch_lora_stream(LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream, LaunchInfo *info) {
    const void *fn = lora_kernel_stream();
    cudaError_t e = encoder();  // the tensor-map encoder, resolved on first use
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    StreamParams k;
    memset(&k, 0, sizeof k);
    k.p = p;
    k.max_segments = bi.max_segments;
    k.runcap = std::max(1, std::min(bi.max_segments, bi.max_loras + std::max(bi.max_bs, 1)));
    const size_t budget = 227 * 1024;
    // base slots: a multiple of the epilogue teams (each slot's barriers are
    // then waited on by one team only), as many as fit
    int Sy = 16 / kStBoxes / kStTeams * kStTeams;
    size_t smem = carve_stream(k, Sy);
    while (smem > budget && Sy > kStTeams) smem = carve_stream(k, Sy -= kStTeams);
    if (smem > budget) return cudaErrorInvalidConfiguration;
    e = ensure_attrs(fn, dev, 1);
    if (e != cudaSuccess) return e;
    int res = 0;
    e = resident(fn, dev, 1, smem, &res, kStThreads);
    if (e != cudaSuccess) return e;
    if (res < 1) return cudaErrorInvalidConfiguration;

    const int s = p.num_tokens;
    const int slots = std::max(1, std::min(std::max(bi.bs, 1), bi.num_loras > 0 ? bi.num_loras : bi.max_loras));
    // tiles are cut at slot runs and at request boundaries: about half a
    // partial tile for each
    const int tiles_est = (s + 127) / 128 + (slots + std::max(bi.bs, 1)) / 2;
    const int tiles_ub = (s + 127) / 128 + std::max(bi.bs, 1) + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    const int64_t ncols = p.off[p.c] - p.off[0];
    // at least 16 R columns: each unit reads h of its tile once (up to four
    // partial-sum planes of 128 x R floats), small next to its base rows
    int64_t cb = (int64_t)tiles_est * ncols / ((int64_t)16 * res);
    cb = std::max<int64_t>(std::max(512, 16 * p.R), (cb + 63) / 64 * 64);
    k.cb = (int)std::min<int64_t>(cb, 1 << 30);
    k.upt = 0;
    for (int j = 0; j < p.c; ++j) k.upt += (p.off[j + 1] - p.off[j] + k.cb - 1) / k.cb;
    if (k.upt == 0) return cudaSuccess;  // no columns
    const int64_t units_ub = (int64_t)tiles_ub * k.upt;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(res, units_ub));

    const int L = bi.max_loras;
    bool ok = true;
    for (int j = 0; j < kMaxSlices; ++j) {
        const int jj = j < p.c ? j : 0;
        ok = ok && encode_2d(&k.tmB[j], p.Bs[jj], (uint64_t)p.R, (uint64_t)L * p.b_rows[jj], (uint64_t)p.R * 2, p.R,
                             64, swizzle_for_row_bytes(p.R * 2));  // one box per 64 columns of a stage
    }
    for (int l = 0; l < kRowBoxLevels; ++l)
        ok = ok && encode_2d(&k.tmY[l], p.y, (uint64_t)p.N, (uint64_t)s, (uint64_t)p.N * 2, 64, 128u >> l,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmYs, p.y, (uint64_t)p.N, (uint64_t)s, (uint64_t)p.N * 2, 64, 32,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && encode_2d(&k.tmYg, p.y, (uint64_t)p.N, (uint64_t)s, (uint64_t)p.N * 2, 64, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kStThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    set_dependent_launch(&attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (info) {
        info->tm = 128;
        info->crmax = p.R;
        info->cluster = 1;
        info->grid = grid;
        info->smem = smem;
    }
    void *args[1] = {&k};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Slot runs of at most 16 tokens on average.
bool wide_runs(const LoraParams &p, const csgmv_batch_info &bi) {
    const int slots = std::max(1, std::min(std::max(bi.bs, 1), bi.num_loras > 0 ? bi.num_loras : bi.max_loras));
    return p.num_tokens / slots <= 16;
}

// Expand-only launch onto a wide output (a vocabulary-wide lm_head) on the
// warp-specialized wide kernel (lora_wide.cuh), on 16-token tiles (32-token
// tiles need twice the accumulators and measured slower).  A tile streams all
// of its slot's B rows, so a slot of up to 16 tokens reads them once.
cudaError_t launch_lora_wide(LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream, LaunchInfo *info) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int slots = std::max(1, std::min(std::max(bi.bs, 1), bi.num_loras > 0 ? bi.num_loras : bi.max_loras));
    const int tm = 16;
    const int rmax = p.R <= 16 ? 16 : (p.R <= 32 ? 32 : 64);
    const void *fn = lora_kernel_wide(tm, rmax);
    if (!fn) return cudaErrorInvalidValue;
    WideParams k;
    memset(&k, 0, sizeof k);
    k.p = p;
    k.max_segments = bi.max_segments;
    k.runcap = std::max(1, std::min(bi.max_segments, bi.max_loras + std::max(bi.max_bs, 1)));
    // tiles by slot when the grouped table fits its share of shared memory
    k.nslot = std::max(1, p.max_loras);
    k.segcap = std::max(1, bi.max_segments);
    k.tokcap = std::max(1, p.num_tokens);
    k.grouped = wide_group_ints(k.nslot, k.segcap, k.tokcap) * 4 <= (size_t)kWideGroupBytes;
    const size_t table_ints = std::max<size_t>((size_t)5 * k.runcap + 1 + 32,
                                               k.grouped ? wide_group_ints(k.nslot, k.segcap, k.tokcap) : 0);
    const size_t budget = 227 * 1024;
    const size_t hf_bytes = (size_t)2 * kWideHfInts * 4 + 2 * 32 * 4;  // h fragments and tokens, two buffers
    const size_t fixed = align_up(3 * 8 * 8 + 32 + table_ints * 4 + 16 + hf_bytes, 1024) + 1024;
    // 512-column stages when four of them fit, else 256
    for (int nt = 512; nt >= 256; nt -= 256) {
        k.nt = nt;
        k.ypitch = nt * 2 + 16;
        k.b_off = (int)align_up((size_t)tm * k.ypitch, 1024);
        k.stage_bytes = (int)align_up((size_t)k.b_off + (size_t)nt * p.R * 2, 1024);
        k.S = (int)std::min<size_t>(8, budget > fixed ? (budget - fixed) / k.stage_bytes : 0);
        if (k.S >= 4) break;
    }
    if (k.S < 2) return cudaErrorInvalidConfiguration;
    k.o_bar = 0;
    k.o_hbar = (int)align_up((size_t)3 * k.S * 8, 16);
    k.o_run = (int)align_up((size_t)k.o_hbar + 4 * 8, 16);
    k.o_hf = (int)align_up((size_t)k.o_run + table_ints * 4, 16);
    k.o_ring = (int)align_up((size_t)k.o_hf + hf_bytes, 1024);
    const size_t smem = (size_t)k.o_ring + (size_t)k.S * k.stage_bytes + 1024;
    // columns per unit: about six units per SM over the expected tiles
    const int64_t ncols = p.off[p.c] - p.off[0];
    const int tiles_est = std::max(slots, (p.num_tokens + tm - 1) / tm);
    int64_t cb = (int64_t)tiles_est * ncols / ((int64_t)6 * sms);
    cb = std::max<int64_t>(k.nt, (cb + k.nt - 1) / k.nt * k.nt);
    k.cb = (int)std::min<int64_t>(cb, (ncols + k.nt - 1) / k.nt * k.nt);
    const int nblk = (int)((ncols + k.cb - 1) / k.cb);
    const int tiles_ub = (p.num_tokens + tm - 1) / tm + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sms, (int64_t)tiles_ub * nblk));
    if (!encode_b_maps(&k.tmB, k.tmBs, p, bi.max_loras, 256)) return cudaErrorInvalidValue;
    if ((e = ensure_attrs(fn, dev, 1)) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    set_dependent_launch(&attr[0]);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kWideThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (info) {
        info->tm = tm;
        info->crmax = rmax;
        info->cluster = 1;
        info->grid = grid;
        info->smem = smem;
    }
    void *args[1] = {&k};
    if ((e = cudaLaunchKernelExC(&cfg, fn, args)) != cudaSuccess) return e;
    return cudaGetLastError();
}

// Token tile for a batch: 16 for one or two tokens per slot run, 32 for a few,
// 128 for prefill.
int token_tile(const LoraParams &p, const csgmv_batch_info &bi) {
    const int slots = std::max(1, std::min(std::max(bi.bs, 1), bi.num_loras > 0 ? bi.num_loras : bi.max_loras));
    const int tps = p.num_tokens / slots;  // mean tokens per slot run
    return tps <= 16 ? 16 : (tps <= 48 ? 32 : 128);
}

// Decode-shaped batches the cluster-free decode kernels take: short slot
// runs, outputs narrower than a vocabulary, and batch-info capacities within
// the kernels' one-round tables.
bool decode_fits(const LoraParams &p, const csgmv_batch_info &bi) {
    return token_tile(p, bi) <= 32 && p.off[p.c] - p.off[0] < kWideCols && p.accumulate &&
           bi.max_segments <= kDecSegCap && bi.max_loras <= kDecLoraCap && p.num_tokens <= kDecPermCap;
}

bool qkv_split_pays(const LoraParams &p, const csgmv_batch_info &bi) {
    const int tm = token_tile(p, bi);
    // Vocabulary-wide outputs on 16- / 32-token tiles: the fused kernel gives
    // each tile's columns to one cluster, which leaves SMs idle and makes every
    // CTA stream tens of thousands of columns; with h in the workspace, the
    // expand-only launch spreads column blocks of every tile over all SMs.
    // Other decode shapes: the split-K shrink and the expand of the decode
    // kernels, which need no cluster barrier.
    if (tm <= 32) return p.off[p.c] - p.off[0] >= kWideCols || decode_fits(p, bi);
    // 128-token tiles: the streaming tcgen05 shrink and expand
    return tm == 128 && p.R >= 16;
}

int qkv_max_parts(const LoraParams &p, const csgmv_batch_info &bi) {
    return decode_fits(p, bi) ? kDecMaxParts : kMaxKParts;
}

int qkv_path(const LoraParams &p, const csgmv_batch_info &bi, size_t workspace_bytes) {
    const size_t hbytes = (size_t)p.num_tokens * p.c * p.R * 4;
    if (p.num_tokens <= 0 || workspace_bytes < kWsHeader + hbytes || !qkv_split_pays(p, bi)) return CSGMV_PATH_FUSED;
    if (decode_fits(p, bi)) return CSGMV_PATH_DECODE;
    if (token_tile(p, bi) == 128 && p.R >= 16) return CSGMV_PATH_STREAM;
    return CSGMV_PATH_SMALL_SPLIT;
}

// The decode kernels (lora_decode.cuh) through the workspace: the split-K
// shrink over one CTA per SM, then the expand as its programmatic dependent.
cudaError_t launch_qkv_decode(LoraParams &ps, LoraParams &pe, const csgmv_batch_info &bi, cudaStream_t stream,
                              void *workspace, size_t workspace_bytes) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int L = bi.max_loras;
    const int cR = ps.c * ps.R;
    const size_t plane = (size_t)ps.num_tokens * ps.ldh;
    const size_t room = workspace_bytes > kWsHeader ? workspace_bytes - kWsHeader : 0;
    const int max_parts = (int)std::max<size_t>(1, std::min<size_t>(kDecMaxParts, plane ? room / (plane * 4) : 1));
    float *planes = reinterpret_cast<float *>(static_cast<char *>(workspace) + kWsHeader);
    const int nkc = (int)((ps.K + 63) / 64);

    // ---- shrink: the table, then A boxes and x rows of up to kc_max chunks
    DecodeParams ks;
    memset(&ks, 0, sizeof ks);
    ks.p = ps;
    ks.p.h = planes;
    ks.p.h_plane = (int64_t)plane;
    ks.p.h_parts = max_parts;
    ks.max_segments = bi.max_segments;
    ks.tile_cap = (int)(csgmv_tile_table_ints(bi.max_loras, bi.max_tokens) / 4 - 1);
    ks.nkc = nkc;
    ks.shrink_grid = sms;
    ks.a_rows = (int)align_up((size_t)cR, 16);
    // the two kernels share an SM: shrink <= 100 KB, expand <= 120 KB
    const size_t budget_s = 100 * 1024, budget_e = 120 * 1024;
    size_t off = 0;
    auto take = [&](size_t bytes, size_t align) {
        off = align_up(off, align);
        const size_t o = off;
        off += bytes;
        return (int)o;
    };
    ks.o_bar = take(16, 16);
    ks.o_tab = take((size_t)kDecTabInts * 4, 16);
    const size_t fixed_s = align_up(off, 1024) + 1024 + (size_t)kDecTM * 16 + 16;
    const size_t per_chunk = (size_t)ks.a_rows * 128 + (size_t)kDecTM * 128;
    ks.kc_max = (int)std::max<size_t>(1, std::min<size_t>(nkc, budget_s > fixed_s ? (budget_s - fixed_s) / per_chunk : 1));
    ks.xpitch = ks.kc_max * 128 + 16;
    ks.o_a = take((size_t)ks.kc_max * ks.a_rows * 128, 1024);
    ks.o_x = take((size_t)kDecTM * ks.xpitch, 16);
    const size_t smem_s = off + 1024;  // slack for aligning the window to 1024 bytes
    if (!encode_2d(&ks.tmA, ps.A, (uint64_t)ps.K, (uint64_t)L * cR, (uint64_t)ps.K * 2, 64, ks.a_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    ks.tmB = ks.tmA;
    for (int j = 0; j < kMaxSlices; ++j) ks.tmBs[j] = ks.tmA;

    // ---- expand: the table, base rows and B rows of up to cols_max columns, h
    DecodeParams ke = ks;
    ke.p = pe;
    ke.p.h = planes;
    ke.p.h_plane = (int64_t)plane;
    ke.p.h_parts = max_parts;
    const int rmax = pe.R <= 16 ? 16 : (pe.R <= 32 ? 32 : 64);
    off = 0;
    ke.o_bar = take(16, 16);
    ke.o_tab = take((size_t)kDecTabInts * 4, 16);
    // h as A fragments: slices x 16-row tiles x k16 steps x (hi, lo) x 512 bytes
    const size_t hs_bytes = (size_t)kMaxSlices * (kDecTM / 16) * (rmax / 16) * 2 * 512;
    const size_t fixed_e = align_up(off, 1024) + 1024 + hs_bytes + (size_t)kDecTM * 16 + 32;
    const size_t per_blk = (size_t)kDecTM * 128 + (size_t)64 * pe.R * 2;
    const int blks = (int)std::max<size_t>(1, std::min<size_t>(8, budget_e > fixed_e ? (budget_e - fixed_e) / per_blk : 1));
    ke.cols_max = 64 * blks;
    ke.ypitch = ke.cols_max * 2 + 16;
    ke.o_y = take((size_t)kDecTM * ke.ypitch, 16);
    ke.o_b = take((size_t)ke.cols_max * pe.R * 2, 1024);
    ke.o_h = take(hs_bytes, 16);
    const size_t smem_e = off + 1024;
    if (!encode_b_maps(&ke.tmB, ke.tmBs, pe, L, 64)) return cudaErrorInvalidValue;
    ke.tmA = ke.tmB;

    const void *fs = lora_kernel_decode(0, rmax), *fe = lora_kernel_decode(1, rmax);
    if (!fs || !fe) return cudaErrorInvalidValue;
    if ((e = ensure_attrs(fs, dev, 1)) != cudaSuccess) return e;
    if ((e = ensure_attrs(fe, dev, 1)) != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    set_dependent_launch(&attr[0]);
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kDecThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(sms, 1, 1);
    cfg.dynamicSmemBytes = smem_s;
    void *args_s[1] = {&ks};
    if ((e = cudaLaunchKernelExC(&cfg, fs, args_s)) != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem_e;
    cfg.blockDim = dim3(kDecExpThreads, 1, 1);
    void *args_e[1] = {&ke};
    if ((e = cudaLaunchKernelExC(&cfg, fe, args_e)) != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_qkv_split(LoraParams &ps, LoraParams &pe, const csgmv_batch_info &bi, cudaStream_t stream,
                             void *workspace, size_t workspace_bytes, int path) {
    if (path == CSGMV_PATH_DECODE) return launch_qkv_decode(ps, pe, bi, stream, workspace, workspace_bytes);
    // the workspace: a header (the part count), then planes of s * c * R floats
    int *header = static_cast<int *>(workspace);
    float *planes = reinterpret_cast<float *>(static_cast<char *>(workspace) + kWsHeader);
    const size_t plane = (size_t)ps.num_tokens * ps.ldh;
    const size_t room = workspace_bytes > kWsHeader ? workspace_bytes - kWsHeader : 0;
    const int max_parts = (int)std::max<size_t>(1, std::min<size_t>(kMaxKParts, plane ? room / (plane * 4) : 1));
    ps.h = planes;
    pe.h = planes;
    pe.h_plane = (int64_t)plane;
    cudaError_t e;
    if (path == CSGMV_PATH_STREAM) {
        ps.h_plane = (int64_t)plane;
        e = launch_lora_sshrink(ps, bi, stream, nullptr, max_parts, header);
        pe.h_parts = max_parts;
        pe.h_parts_dev = header;
    } else {
        e = launch_lora(kModeShrink, ps, bi, stream, nullptr);
        pe.h_parts = 1;
        pe.h_parts_dev = nullptr;
    }
    if (e != cudaSuccess) return e;
    return launch_lora(kModeExpand, pe, bi, stream, nullptr);
}

cudaError_t launch_lora(int mode, LoraParams &p, const csgmv_batch_info &bi, cudaStream_t stream,
                        LaunchInfo *info) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const int cR = p.c * p.R;
    const int rmax = p.R <= 16 ? 16 : (p.R <= 32 ? 32 : 64);
    const int s = p.num_tokens;
    const int tm = token_tile(p, bi);
    // Prefill tiles expand on tcgen05 when every slice edge and the B rows
    // suit its operand layouts (16-column pieces, 32..128-byte swizzled rows).
    bool tc = tm == 128 && mode != kModeShrink && p.R >= 16;
    for (int j = 0; j <= p.c; ++j) tc = tc && p.off[j] % 16 == 0;
    // Shrink-only calls on 128-token tiles of moderate K run on the
    // warp-specialized kernel (one CTA per tile, whole K, tcgen05); the fused
    // and expand calls measure faster on the cluster kernel.
    // Shrink-only calls on 128-token tiles run on the streaming tcgen05
    // shrink (h itself: one part of K).
    if (tm == 128 && p.R >= 16 && mode == kModeShrink) return launch_lora_sshrink(p, bi, stream, info, 1, nullptr);
    // Expand-only calls on 128-token tiles stream base through the
    // warp-specialized tcgen05 expand.
    if (tm == 128 && p.R >= 16 && mode == kModeExpand) return launch_lora_stream(p, bi, stream, info);
    // Expand-only calls of short slot runs (at most 16 tokens a slot on
    // average: an lm_head decode or pruned lm_head pass) onto a
    // vocabulary-wide output: the warp-specialized wide kernel.  Longer runs
    // take the small-tile kernel's 512-column stages.
    if (mode == kModeExpand && tm <= 32 && p.off[p.c] - p.off[0] >= kWideCols && wide_runs(p, bi))
        return launch_lora_wide(p, bi, stream, info);
    if (tm <= 32) {
        const cudaError_t es = launch_lora_small(mode, p, bi, stream, info, rmax, tm);
        if (es != cudaErrorInvalidConfiguration) return es;
    }
    const void *fn = mode == kModeFused ? lora_kernel_fused(tm, rmax, tc)
                   : mode == kModeShrink ? lora_kernel_shrink(tm, rmax, tc)
                                         : lora_kernel_expand(tm, rmax, tc);
    if (!fn) return cudaErrorInvalidValue;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;

    TmaKernelParams k;
    memset(&k, 0, sizeof k);
    k.p = p;
    k.max_segments = bi.max_segments;
    k.runcap = std::max(1, std::min(bi.max_segments, bi.max_loras + std::max(bi.max_bs, 1)));
    k.ah_slices = p.c;  // until the column split is known
    const size_t budget = 227 * 1024;
    const int nkc = (int)((p.K + 63) / 64);
    const int nb64 = tc ? kTcCols / 64 : (tm >= 128 ? 1 : (tm >= 64 ? 2 : 4));
    const int ntile_cols = 64 * nb64;

    // Cluster size: 8 unless a smaller cluster covers clearly more SMs.  Ring
    // depths: decode tiles put every stage of a CTA in flight at once, prefill
    // tiles get as many stages as shared memory holds (up to 8).
    int cs_pick[3] = {0, 0, 0}, res_pick[3] = {0, 0, 0}, s1_pick[3] = {0, 0, 0}, s2_pick[3] = {0, 0, 0};
    const int cs_list[3] = {8, 4, 2};  // at most 8: the reduce sums up to eight peers
    const int ncand = mode == kModeExpand ? 1 : 3;
    int best_sms = 0;
    for (int ci = 0; ci < ncand; ++ci) {
        const int cs = mode == kModeExpand ? 1 : cs_list[ci];
        if (tm % cs) continue;
        const int kc_per = (nkc + cs - 1) / cs;
        const int cols_per = (p.off[p.c] - p.off[0] + cs - 1) / cs;
        const int tiles_per = std::max(1, (cols_per + ntile_cols - 1) / ntile_cols);
        int S1 = tm <= 32 ? std::min(16, std::max(2, kc_per)) : std::min(4, std::max(2, kc_per));
        int S2 = tm <= 32 ? std::min(8, std::max(2, tiles_per + 1)) : 8;
        if (tc) {  // shrink stages that fit where the h operand tiles go anyway
            const int sh_stage = (int)align_up((size_t)tm * 128 + align_up((size_t)cR, 16) * 128, 1024);
            S1 = std::max(2, std::min(kc_per, (int)((size_t)p.c * 2 * kTcAhBytes / sh_stage)));
            S2 = 4;
        }
        size_t smem = carve(k, mode, tm, cs, S1, S2, tc);
        while (smem > budget && (S1 > 2 || S2 > 2)) {
            if (S2 > 4 || (S2 > 2 && S1 <= 2)) --S2; else --S1;
            smem = carve(k, mode, tm, cs, S1, S2, tc);
        }
        if (smem > budget) continue;
        e = ensure_attrs(fn, dev, cs);
        if (e != cudaSuccess) return e;
        int res = 0;
        if (resident(fn, dev, cs, smem, &res) != cudaSuccess) continue;
        cs_pick[ci] = cs; res_pick[ci] = res; s1_pick[ci] = S1; s2_pick[ci] = S2;
        best_sms = std::max(best_sms, res * cs);
    }
    int pick = -1;
    for (int ci = 0; ci < ncand; ++ci)
        if (cs_pick[ci] && res_pick[ci] * cs_pick[ci] * 100 >= best_sms * 85) { pick = ci; break; }
    if (pick < 0) return cudaErrorInvalidConfiguration;
    const int cs = cs_pick[pick];
    const int best_res = res_pick[pick];
    size_t smem = carve(k, mode, tm, cs, s1_pick[pick], s2_pick[pick], tc);

    // Column blocks per tile when the tiles alone cannot fill the machine.
    const int tiles_ub = (s + tm - 1) / tm + std::min(std::max(bi.bs, 1), std::max(bi.max_loras, 1));
    if (mode == kModeShrink) {
        k.p.nsplit = 1;
    } else {
        const int nblk = (p.off[p.c] - p.off[0] + 63) / 64;
        const int max_split = std::max(1, nblk / (cs * nb64));
        k.p.nsplit = std::max(1, std::min(best_res / std::max(tiles_ub, 1), max_split));
    }
    if (tc && mode == kModeExpand && p.c > 1) {
        // At least one column block per slice, so that a CTA's columns mostly
        // stay within one slice: then the h operand tiles of fewer slices are
        // needed, and the room goes to more expand stages in flight.
        const int nblk = (p.off[p.c] - p.off[0] + 63) / 64;
        k.p.nsplit = std::max(k.p.nsplit, std::min(p.c, std::max(1, nblk / nb64)));
        k.ah_slices = max_slice_span(k.p, k.p.nsplit * cs);
        int S2 = 8;
        smem = carve(k, mode, tm, cs, 1, S2, tc);
        while (smem > budget && S2 > 2) smem = carve(k, mode, tm, cs, 1, --S2, tc);
        if (smem > budget) return cudaErrorInvalidConfiguration;
    } else if (tc) {
        k.ah_slices = max_slice_span(k.p, k.p.nsplit * cs);
        if (k.ah_slices < p.c) smem = carve(k, mode, tm, cs, k.S1, k.S2, tc);
    }
    const int64_t units_ub = (int64_t)tiles_ub * k.p.nsplit;
    const int nclusters = (int)std::max<int64_t>(1, std::min<int64_t>(best_res, units_ub));

    // TMA descriptors for the weight tiles: one box per shrink chunk (all c*R
    // rows of a slot, 64 wide) and one per expand tile (NT rows of B, all R
    // columns).  Unused ones point at a valid tensor.
    const int L = bi.max_loras;
    const int nt = 64 * nb64;
    bool ok = true;
    if (mode != kModeExpand)
        ok = ok && encode_2d(&k.tmA, p.A, (uint64_t)p.K, (uint64_t)L * cR, (uint64_t)p.K * 2, 64, k.a_rows,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    if (mode != kModeShrink)
        ok = ok && encode_b(k, L, nt);
    if (mode == kModeExpand) k.tmA = k.tmB;
    if (mode == kModeShrink) k.tmB = k.tmA;
    // row boxes of x and base for 128-token tiles of consecutive tokens
    k.row_tma = tm == 128 ? 1 : 0;
    if (k.row_tma && mode != kModeExpand)
        ok = ok && encode_2d(&k.tmX, p.x, (uint64_t)p.K, (uint64_t)s, (uint64_t)p.K * 2, 64, tm,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    else
        k.tmX = k.tmA;
    if (k.row_tma && mode != kModeShrink)  // base loads (accumulating) and whole-tile stores
        ok = ok && encode_2d(&k.tmY, p.y, (uint64_t)p.N, (uint64_t)s, (uint64_t)p.N * 2, 64, tm,
                             CU_TENSOR_MAP_SWIZZLE_128B);
    else
        k.tmY = k.tmA;
    k.tmXg = k.tmA;  // the cluster kernel gathers rows with cp.async
    if (!ok) return cudaErrorInvalidValue;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nclusters * cs, 1, 1);
    cfg.blockDim = dim3(kTmaThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_dependent_launch(&attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (info) {
        info->tm = tm;
        info->crmax = rmax;
        info->cluster = cs;
        info->grid = nclusters * cs;
        info->smem = smem;
    }
    void *args[1] = {&k};
    e = cudaLaunchKernelExC(&cfg, fn, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csgmv
