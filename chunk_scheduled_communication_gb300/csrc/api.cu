// api.cu -- the C ABI of libsyn (see include/syn.h for the contract).
//
// Host side of the chunk-scheduled operators: plan creation (schedule build,
// device tables, flags, counters, receive buffers), tensor-map encoding, and
// the per-call orchestration of the staging backends of the Syncopate summary
// page (method ¶3, paper §5.2, Fig. 7):
//   CE            side streams (chunks round-robin in arrival order, so several
//                 copy engines run at once): per chunk, cudaMemcpyAsync then a
//                 stream-ordered flag write (cuStreamWriteValue32, which fences
//                 prior writes), concurrent with the fused kernel on the caller's
//                 stream
//   TMA_DEDICATED comm_sms extra CTAs of the same cooperative grid copy chunks
//   TMA_COLOCATED a staging warp in every GEMM CTA copies chunk slices
//   LDST_DEDICATED / LDST_COLOCATED  the same placements, copying with warp-wide
//                 16-byte vector loads and stores instead of TMA bulk copies
//   TMA_COLOCATED_SMEM  GEMM-RS/AR: peers fetched per tile into shared memory
//   UNFUSED       whole staging copy, then the same kernel without waits
//   DECOMPOSED    one kernel launch per chunk group after its copies (the
//                 split multi-kernel baseline of paper Fig. 2(b))
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "fused.h"
#include "host_util.h"
#include "schedule.h"
#include "syn.h"

using namespace syn;

namespace {

thread_local std::string g_err;

int fail(int code, const std::string &msg) {
    g_err = msg;
    return code;
}

#define SYN_CK(call)                                                                       \
    do {                                                                                   \
        cudaError_t e__ = (call);                                                          \
        if (e__ != cudaSuccess)                                                            \
            return fail(SYN_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e__)); \
    } while (0)

PFN_cuTensorMapEncodeTiled_v12000 p_encode = nullptr;
PFN_cuStreamWriteValue32_v11070 p_write32 = nullptr;
std::once_flag g_drv_once;
std::string g_drv_err;

int load_driver() {
    std::call_once(g_drv_once, [] {
        cudaDriverEntryPointQueryResult q;
        void *fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            g_drv_err = "cuTensorMapEncodeTiled is not available";
            return;
        }
        p_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 11070, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr) {
            g_drv_err = "cuStreamWriteValue32 is not available";
            return;
        }
        p_write32 = reinterpret_cast<PFN_cuStreamWriteValue32_v11070>(fn);
    });
    if (p_encode == nullptr || p_write32 == nullptr) return fail(SYN_ERR_CUDA, g_drv_err);
    return SYN_OK;
}

uint64_t env_timeout_ns() {
    const char *s = std::getenv("SYN_TIMEOUT_NS");
    if (s != nullptr && *s) {
        const unsigned long long v = std::strtoull(s, nullptr, 10);
        if (v > 0) return v;
    }
    return 2000000000ull;
}

// 2-D tiled tensor map over a row-major matrix [rows, cols].
int encode_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols,
              uint64_t rows, uint32_t box_cols, uint32_t box_rows,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * (uint64_t)esize};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = p_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SYN_ERR_CUDA, "cuTensorMapEncodeTiled failed: " + std::to_string((int)r));
    return SYN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace syn {
int host_fail(int code, const std::string &msg) { return fail(code, msg); }
int host_load_driver() { return load_driver(); }
int host_encode_2d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, uint64_t cols,
                   uint64_t rows, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swz) {
    return encode_2d(m, base, dt, esize, cols, rows, box_cols, box_rows, swz);
}
CUresult host_write32(cudaStream_t st, uint32_t *addr, uint32_t value) {
    return p_write32(reinterpret_cast<CUstream>(st), reinterpret_cast<CUdeviceptr>(addr), value,
                     CU_STREAM_WRITE_VALUE_DEFAULT);
}
uint64_t host_timeout_ns() { return env_timeout_ns(); }
}  // namespace syn

void syn::set_last_error(const std::string &msg) { g_err = msg; }

struct syn_plan_s {
    Schedule s;
    syn_knobs_t kn;
    int device = 0, num_sms = 0;
    int grid_compute = 0, grid_comm = 0, smem = 0;
    int resident = 0;                              // CTAs that fit on the device at once
    LaunchCfg lc = {256, 64, 4, false, false, 0};  // compiled kernel instance
    uint32_t epoch = 0;
    // device state
    int32_t *d_tiles = nullptr, *d_transfers = nullptr, *d_err = nullptr;
    uint32_t *d_in_flags = nullptr, *d_in_cnt = nullptr, *d_out_flags = nullptr, *d_out_cnt = nullptr;
    unsigned long long *d_stats = nullptr;
    unsigned long long *d_trace = nullptr;  // trace = 2: [n_tiles][5] stamps + walker
    uint8_t *d_recv = nullptr;
    uint64_t recv_bytes = 0;
    float *d_red = nullptr;                 // RED: fp32 partials of the reducing tiles
    size_t red_bytes = 0;
    float *d_push = nullptr;                // dedicated push: send rows as produced [M, N]
    int32_t *d_push_list = nullptr;         // dedicated push: send row chunks, production order
    int n_push = 0;
    int64_t recv_slot_rows = 0;
    cudaStream_t side = nullptr;            // side stream 0 (DECOMPOSED copies; CE stream 0)
    std::vector<cudaStream_t> ce_side;      // CE: transfers go round-robin over these
    std::vector<cudaEvent_t> ce_join;       // CE: one join event per side stream
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    std::vector<cudaEvent_t> ev_transfer;  // DECOMPOSED: one per transfer
    std::vector<std::pair<int, int>> groups;  // DECOMPOSED: tile-list ranges of equal key
    std::vector<int> group_key;
    // tensor-map cache
    TensorMaps maps;
    std::vector<const void *> map_key;
};

namespace {

bool staged_peers(const syn_plan_s *pl) {
    return pl->s.op != SYN_OP_AG_GEMM && pl->kn.backend != SYN_BACKEND_TMA_COLOCATED_SMEM;
}

void free_plan(syn_plan_s *pl) {
    if (pl == nullptr) return;
    if (pl->side) cudaStreamSynchronize(pl->side);
    for (cudaStream_t x : pl->ce_side)
        if (x != pl->side) cudaStreamSynchronize(x);
    cudaFree(pl->d_tiles);
    cudaFree(pl->d_transfers);
    cudaFree(pl->d_err);
    cudaFree(pl->d_in_flags);
    cudaFree(pl->d_in_cnt);
    cudaFree(pl->d_out_flags);
    cudaFree(pl->d_out_cnt);
    cudaFree(pl->d_stats);
    cudaFree(pl->d_trace);
    cudaFree(pl->d_recv);
    cudaFree(pl->d_red);
    cudaFree(pl->d_push);
    cudaFree(pl->d_push_list);
    for (cudaEvent_t e : pl->ev_transfer) cudaEventDestroy(e);
    if (pl->ev_fork) cudaEventDestroy(pl->ev_fork);
    if (pl->ev_join) cudaEventDestroy(pl->ev_join);
    for (cudaEvent_t e : pl->ce_join) cudaEventDestroy(e);
    for (cudaStream_t x : pl->ce_side)
        if (x != pl->side) cudaStreamDestroy(x);
    if (pl->side) cudaStreamDestroy(pl->side);
    delete pl;
}

// A2A-GEMM plans are AG-GEMM plans over per-source row blocks of their own
// size (no uniform M/R).
bool is_a2a(const Schedule &s) { return s.op == SYN_OP_AG_GEMM && s.M_r == 0; }

void fill_info(const Schedule &s, const syn_knobs_t &kn, syn_plan_info_t *info) {
    std::memset(info, 0, sizeof(*info));
    info->op = s.op;
    info->R = s.R;
    info->rank = s.rank;
    info->backend = kn.backend;
    info->order = s.order;
    info->M = s.M;
    info->N = s.N;
    info->K = s.K;
    info->M_r = s.M_r;
    info->chunk_rows = s.cr;
    info->split = s.split;
    info->n_row_chunks = s.n_rc;
    info->n_transfers = (int)s.transfers.size();
    info->tile_m = s.tile_m;
    info->tile_n = s.tile_n;
    info->tiles_m = s.tiles_m;
    info->tiles_n = s.tiles_n;
    info->n_tiles = s.n_tiles;
    info->a2a = is_a2a(s) ? 1 : 0;
}

syn_knobs_t resolve_knobs(const syn_knobs_t *k) {
    syn_knobs_t kn;
    syn_knobs_default(&kn);
    if (k != nullptr) kn = *k;
    if (kn.tile_m == 0) kn.tile_m = 128;
    if (kn.tile_n == 0) kn.tile_n = 256;
    if (kn.group_m <= 0) kn.group_m = 8;
    if (kn.slice_kb <= 0) kn.slice_kb = 128;
    if (kn.timeout_ns == 0) kn.timeout_ns = env_timeout_ns();
    return kn;
}

// Common parameter block of one call.
KernelParams base_params(syn_plan_s *pl) {
    const Schedule &s = pl->s;
    KernelParams p;
    std::memset(&p, 0, sizeof(p));
    p.op = s.op;
    p.R = s.R;
    p.rank = s.rank;
    p.M = (int32_t)s.M;
    p.N = (int32_t)s.N;
    p.K = (int32_t)s.K;
    p.M_r = (int32_t)s.M_r;
    p.cr = (int32_t)s.cr;
    p.split = s.split;
    p.rb = s.rb;
    p.n_rc = s.n_rc;
    p.tiles_m = s.tiles_m;
    p.tiles_n = s.tiles_n;
    p.t_begin = 0;
    p.t_end = s.n_tiles;
    p.G = pl->grid_compute;
    p.n_comm = 0;
    p.colocated = 0;
    p.waits = 1;
    p.drop_transfer = pl->kn.debug_drop_chunk;
    p.delay_transfer = pl->kn.debug_delay_us > 0 ? pl->kn.debug_delay_chunk : -1;
    p.delay_ns = (uint32_t)std::min<int64_t>((int64_t)pl->kn.debug_delay_us * 1000, 4000000000ll);
    p.epoch = pl->epoch;
    p.timeout_ns = pl->kn.timeout_ns;
    p.tile_list = pl->d_tiles;
    p.transfers = pl->d_transfers;
    p.n_transfers = (int32_t)s.transfers.size();
    p.in_flags = pl->d_in_flags;
    p.in_cnt = pl->d_in_cnt;
    p.out_flags = pl->d_out_flags;
    p.out_cnt = pl->d_out_cnt;
    p.err = pl->d_err;
    p.stats = pl->kn.trace ? pl->d_stats : nullptr;
    p.trace = pl->d_trace;
    return p;
}

// Operand tensor maps for the plan's kernel instance: A / gathered [M, K] in
// boxes of tile_k x 128 rows (128-byte swizzle at tile_k 64, 64-byte at 32),
// B [K, N] in boxes of 64 columns x tile_k rows (128-byte swizzle).
int encode_operands(syn_plan_s *pl, const void *A, const void *B) {
    const Schedule &s = pl->s;
    const int tk = pl->lc.tile_k;
    const CUtensorMapSwizzle a_swz = tk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    int rc = encode_2d(&pl->maps.a, A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.K, s.M, tk, 128, a_swz);
    if (rc != SYN_OK) return rc;
    return encode_2d(&pl->maps.b, B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.N, s.K, 64, tk,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

int finish_params_for_staging(syn_plan_s *pl, KernelParams &p) {
    const int64_t tbytes = (int64_t)p.cr * p.row_bytes;
    int64_t slice = (int64_t)pl->kn.slice_kb * 1024;
    slice = std::max<int64_t>(16, slice & ~int64_t(15));
    if (slice > tbytes) slice = tbytes;
    p.slice_bytes = (int32_t)slice;
    p.slices_per_transfer = (int32_t)((tbytes + slice - 1) / slice);
    return SYN_OK;
}

cudaError_t launch(syn_plan_s *pl, const KernelParams &p, int grid, cudaStream_t st) {
    LaunchCfg lc = pl->lc;
    lc.grid = grid;
    // one kernel per call, nothing else queued before it by this call: its
    // launch and set-up may overlap the previous kernel on the stream (the
    // kernel waits for that grid before it touches global memory)
    const int be = pl->kn.backend;
    lc.overlap_prev = lc.pair && (be == SYN_BACKEND_TMA_DEDICATED || be == SYN_BACKEND_TMA_COLOCATED ||
                                  be == SYN_BACKEND_TMA_COLOCATED_SMEM || be == SYN_BACKEND_LDST_DEDICATED ||
                                  be == SYN_BACKEND_LDST_COLOCATED);
    switch (pl->s.op) {
        case SYN_OP_AG_GEMM: return launch_fused_ag(p, pl->maps, lc, st);
        case SYN_OP_GEMM_RS: return launch_fused_rs(p, pl->maps, lc, st);
        default: return launch_fused_ar(p, pl->maps, lc, st);
    }
}

// Issue the staging copies of all transfers on `st` (CE); optionally a flag
// write after each and/or an event record after each.
int ce_copies(syn_plan_s *pl, const KernelParams &p, const cudaStream_t *streams, int n_streams, bool flags,
              bool events) {
    const Schedule &s = pl->s;
    for (size_t a = 0; a < s.transfers.size(); ++a) {
        // transfer a on stream a mod n: copies in arrival order spread over the
        // copy engines; each flag write follows its own copy in its stream
        cudaStream_t st = streams[a % (size_t)n_streams];
        const int code = s.transfers[a];
        const bool skip = (s.op == SYN_OP_AG_GEMM && p.local_inplace && code % s.R == s.rank);
        if (!skip) {
            const uint8_t *src;
            uint8_t *dst;
            int64_t bytes;
            transfer_span(p, code, src, dst, bytes);
            if (bytes > 0)  // (empty A2A-GEMM chunks still publish their flag)
                SYN_CK(cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyDeviceToDevice, st));
            if (flags && (int)a != p.drop_transfer) {
                CUresult r = p_write32(reinterpret_cast<CUstream>(st),
                                       reinterpret_cast<CUdeviceptr>(pl->d_in_flags + code), p.epoch,
                                       CU_STREAM_WRITE_VALUE_DEFAULT);
                if (r != CUDA_SUCCESS) return fail(SYN_ERR_CUDA, "cuStreamWriteValue32 failed");
            }
        }
        if (events) SYN_CK(cudaEventRecord(pl->ev_transfer[a], st));
    }
    return SYN_OK;
}

// Run one call of the plan's operator once `p` and the maps are filled.
int run(syn_plan_s *pl, KernelParams &p, cudaStream_t st) {
    finish_params_for_staging(pl, p);
    const int be = pl->kn.backend;
    int rc;
    switch (be) {
        case SYN_BACKEND_CE: {
            SYN_CK(cudaEventRecord(pl->ev_fork, st));
            SYN_CK(launch(pl, p, pl->grid_compute, st));
            const int n = (int)pl->ce_side.size();
            for (int i = 0; i < n; ++i) SYN_CK(cudaStreamWaitEvent(pl->ce_side[i], pl->ev_fork, 0));
            if ((rc = ce_copies(pl, p, pl->ce_side.data(), n, true, false)) != SYN_OK) return rc;
            for (int i = 0; i < n; ++i) {
                SYN_CK(cudaEventRecord(pl->ce_join[i], pl->ce_side[i]));
                SYN_CK(cudaStreamWaitEvent(st, pl->ce_join[i], 0));
            }
            return SYN_OK;
        }
        case SYN_BACKEND_LDST_DEDICATED:
        case SYN_BACKEND_TMA_DEDICATED:
            p.ldst = be == SYN_BACKEND_LDST_DEDICATED ? 1 : 0;
            p.n_comm = pl->grid_comm;
            SYN_CK(launch(pl, p, pl->grid_compute + pl->grid_comm, st));
            return SYN_OK;
        case SYN_BACKEND_LDST_COLOCATED:
        case SYN_BACKEND_TMA_COLOCATED:
            p.ldst = be == SYN_BACKEND_LDST_COLOCATED ? 1 : 0;
            p.colocated = 1;
            SYN_CK(launch(pl, p, pl->grid_compute, st));
            return SYN_OK;
        case SYN_BACKEND_TMA_COLOCATED_SMEM:
            p.waits = 0;  // the peers' partials are resident: fetched per tile, no staging
            if (p.push_dedicated) p.n_comm = pl->grid_comm;
            SYN_CK(launch(pl, p, pl->grid_compute + (p.push_dedicated ? pl->grid_comm : 0), st));
            return SYN_OK;
        case SYN_BACKEND_UNFUSED:
            if ((rc = ce_copies(pl, p, &st, 1, false, false)) != SYN_OK) return rc;
            p.waits = 0;
            SYN_CK(launch(pl, p, pl->grid_compute, st));
            return SYN_OK;
        case SYN_BACKEND_DECOMPOSED: {
            SYN_CK(cudaEventRecord(pl->ev_fork, st));
            SYN_CK(cudaStreamWaitEvent(pl->side, pl->ev_fork, 0));
            if ((rc = ce_copies(pl, p, &pl->side, 1, false, true)) != SYN_OK) return rc;
            p.waits = 0;
            for (size_t g = 0; g < pl->groups.size(); ++g) {
                const int key = pl->group_key[g];
                if (key >= 0) SYN_CK(cudaStreamWaitEvent(st, pl->ev_transfer[key], 0));
                KernelParams q = p;
                q.t_begin = pl->groups[g].first;
                q.t_end = pl->groups[g].second;
                const int per = pl->lc.pair ? 2 : 1;
                const int grid = std::min(q.t_end - q.t_begin, pl->resident / per) * per;
                q.G = grid;
                SYN_CK(launch(pl, q, grid, st));
            }
            SYN_CK(cudaEventRecord(pl->ev_join, pl->side));
            SYN_CK(cudaStreamWaitEvent(st, pl->ev_join, 0));
            return SYN_OK;
        }
        default:
            return fail(SYN_ERR_INVALID, "unknown backend");
    }
}

int check_plan(syn_plan_t plan, int op, bool a2a = false) {
    if (plan == nullptr) return fail(SYN_ERR_INVALID, "null plan");
    if (plan->s.op != op || is_a2a(plan->s) != a2a)
        return fail(SYN_ERR_INVALID, "plan was created for another operator");
    return SYN_OK;
}

}  // namespace

// ============================================================================ C ABI

extern "C" {

int syn_knobs_default(syn_knobs_t *k) {
    if (k == nullptr) return fail(SYN_ERR_INVALID, "null knobs");
    std::memset(k, 0, sizeof(*k));
    k->backend = SYN_BACKEND_TMA_COLOCATED;
    k->comm_sms = 8;
    k->tile_m = 128;
    k->tile_n = 256;
    k->group_m = 8;
    k->slice_kb = 128;
    k->timeout_ns = 0;
    k->debug_drop_chunk = -1;
    k->debug_delay_chunk = -1;
    k->trace = 0;
    k->stages = 0;
    k->tile_k = 0;
    return SYN_OK;
}

int syn_schedule_build(syn_op_t op, int R, int rank, const syn_layout_t *layout, int64_t chunk_rows,
                       int split, syn_order_t order, const syn_knobs_t *knobs, syn_plan_info_t *info,
                       int32_t *tile_list, int32_t *tile_key, int32_t *transfers) {
    if (layout == nullptr) return fail(SYN_ERR_INVALID, "null layout");
    const syn_knobs_t kn = resolve_knobs(knobs);
    Schedule s;
    std::string err;
    const int rc = build_schedule(op, R, rank, *layout, chunk_rows, split, order, kn, s, err);
    if (rc != SYN_OK) return fail(rc, err);
    if (info) fill_info(s, kn, info);
    if (tile_list) std::memcpy(tile_list, s.tile_list.data(), s.tile_list.size() * sizeof(int32_t));
    if (tile_key) std::memcpy(tile_key, s.tile_key.data(), s.tile_key.size() * sizeof(int32_t));
    if (transfers) std::memcpy(transfers, s.transfers.data(), s.transfers.size() * sizeof(int32_t));
    return SYN_OK;
}

int syn_device_sms(int *num_sms) {
    if (num_sms == nullptr) return fail(SYN_ERR_INVALID, "null pointer");
    *num_sms = 0;
    int dev = 0;
    SYN_CK(cudaGetDevice(&dev));
    SYN_CK(cudaDeviceGetAttribute(num_sms, cudaDevAttrMultiProcessorCount, dev));
    return SYN_OK;
}

}  // extern "C"

namespace {

// Plan creation shared by syn_plan_create and syn_plan_create_a2a
// (block_rows: the A2A-GEMM per-source row counts, else NULL).
int plan_create(syn_plan_t *out, syn_op_t op, int R, int rank, const syn_layout_t *layout, int64_t chunk_rows,
                int split, syn_order_t order, const syn_knobs_t *knobs, const int64_t *block_rows) {
    if (out == nullptr || layout == nullptr) return fail(SYN_ERR_INVALID, "null argument");
    *out = nullptr;
    int rc = load_driver();
    if (rc != SYN_OK) return rc;
    const syn_knobs_t kn = resolve_knobs(knobs);
    if (kn.backend < SYN_BACKEND_CE || kn.backend > SYN_BACKEND_LDST_COLOCATED)
        return fail(SYN_ERR_INVALID, "unknown backend");
    if (kn.backend == SYN_BACKEND_TMA_COLOCATED_SMEM && op == SYN_OP_AG_GEMM)
        return fail(SYN_ERR_UNSUPPORTED, "TMA_COLOCATED_SMEM applies to GEMM-RS/AR only");
    const bool dedicated = kn.backend == SYN_BACKEND_TMA_DEDICATED || kn.backend == SYN_BACKEND_LDST_DEDICATED;
    if (dedicated && (kn.comm_sms < 1 || kn.comm_sms > 32))
        return fail(SYN_ERR_INVALID, "comm_sms must be in [1, 32]");

    syn_plan_s *pl = new syn_plan_s();
    pl->kn = kn;
    std::string err;
    rc = build_schedule(op, R, rank, *layout, chunk_rows, split, order, kn, pl->s, err, block_rows);
    if (rc != SYN_OK) {
        delete pl;
        return fail(rc, err);
    }
    const Schedule &s = pl->s;
    auto bail = [&](int code, const std::string &msg) {
        free_plan(pl);
        return fail(code, msg);
    };
#define PL_CK(call)                                                                         \
    do {                                                                                    \
        cudaError_t e__ = (call);                                                           \
        if (e__ != cudaSuccess) return bail(SYN_ERR_CUDA, std::string(#call) + ": " + cudaGetErrorString(e__)); \
    } while (0)
    PL_CK(cudaGetDevice(&pl->device));
    PL_CK(cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->device));
    int coop = 0;
    PL_CK(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, pl->device));
    if (!coop) return bail(SYN_ERR_UNSUPPORTED, "device has no cooperative launch");
    pl->lc.tile_n = s.tile_n;
    pl->lc.tile_k = kn.tile_k == 0 ? 64 : kn.tile_k;
    pl->lc.stg = (kn.backend == SYN_BACKEND_TMA_COLOCATED);
    pl->lc.pair = (s.tile_m == 256);
    // resident peers: reducer warps stream the peer sum (default), or the
    // epilogue reduces through a shared-memory peer ring
    pl->lc.red = uses_reducer_warps(s.op, kn, s.tile_n);
    pl->lc.stages = kn.stages > 0 ? kn.stages
                                  : default_stages(s.op, s.tile_n, pl->lc.tile_k, pl->lc.stg, pl->lc.pair,
                                                   pl->lc.red);
    pl->smem = fused_smem_bytes(s.op, pl->lc);
    if (pl->smem < 0)
        return bail(SYN_ERR_UNSUPPORTED,
                    "no compiled kernel for tile_m " + std::to_string(s.tile_m) + ", tile_n " +
                        std::to_string(pl->lc.tile_n) + ", tile_k " + std::to_string(pl->lc.tile_k) +
                        ", stages " + std::to_string(pl->lc.stages) + " with this operator and backend");
    if (kn.direct_fetch && s.op != SYN_OP_AG_GEMM)
        return bail(SYN_ERR_UNSUPPORTED, "direct_fetch applies to AG-GEMM and A2A-GEMM only");
    const bool push_ded = kn.rs_push && kn.push_sms > 0;
    if (kn.push_sms < 0 || kn.push_sms > 32) return bail(SYN_ERR_INVALID, "push_sms must be in [0, 32]");
    if (kn.push_sms > 0 && !kn.rs_push) return bail(SYN_ERR_INVALID, "push_sms needs rs_push = 1");
    if (kn.rs_push && (s.op != SYN_OP_GEMM_RS || epi_tma_rs(pl->lc) != 1))
        return bail(SYN_ERR_UNSUPPORTED,
                    "rs_push needs GEMM-RS with TMA_COLOCATED_SMEM reducer warps and a pipeline depth "
                    "that leaves room for the epilogue's store staging (tile_n 256)");
    // CTAs that can be resident at once: one per SM, or (CTA pairs) twice the
    // co-resident 2-CTA clusters, which may be fewer than SMs / 2
    pl->resident = pl->num_sms;
    if (pl->lc.pair) {
        const int nc = fused_max_clusters(s.op, pl->lc);
        if (nc <= 0) return bail(SYN_ERR_UNSUPPORTED, "2-CTA clusters of this kernel cannot be resident");
        pl->resident = std::min(pl->num_sms, 2 * nc);
    }
    const int cta_per_tile = pl->lc.pair ? 2 : 1;
    if (dedicated || push_ded) {
        const int n = push_ded ? kn.push_sms : kn.comm_sms;
        pl->grid_comm = pl->lc.pair ? (n + 1) / 2 * 2 : n;
        if (pl->grid_comm >= pl->resident) return bail(SYN_ERR_INVALID, "comm_sms >= resident CTAs");
        pl->grid_compute = std::min(s.n_tiles, (pl->resident - pl->grid_comm) / cta_per_tile) * cta_per_tile;
    } else {
        pl->grid_comm = 0;
        pl->grid_compute = std::min(s.n_tiles, pl->resident / cta_per_tile) * cta_per_tile;
    }
    if (s.op == SYN_OP_GEMM_RS && kn.backend == SYN_BACKEND_TMA_COLOCATED_SMEM && kn.reduce_spread == 0)
        spread_reduce_tiles(pl->s, pl->grid_compute / cta_per_tile, pl->lc.red);
    const size_t n_flags = (size_t)s.n_rc * s.R;
    PL_CK(cudaMalloc(&pl->d_tiles, s.tile_list.size() * sizeof(int32_t)));
    PL_CK(cudaMalloc(&pl->d_transfers, std::max<size_t>(1, s.transfers.size()) * sizeof(int32_t)));
    PL_CK(cudaMalloc(&pl->d_err, 4 * sizeof(int32_t)));
    PL_CK(cudaMalloc(&pl->d_in_flags, n_flags * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_in_cnt, 2 * n_flags * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_out_flags, (size_t)s.n_rc * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_out_cnt, 2 * (size_t)s.n_rc * sizeof(uint32_t)));
    PL_CK(cudaMalloc(&pl->d_stats, 2 * sizeof(unsigned long long)));
    PL_CK(cudaMemcpy(pl->d_tiles, s.tile_list.data(), s.tile_list.size() * sizeof(int32_t),
                     cudaMemcpyHostToDevice));
    if (kn.debug_corrupt_entry > 0) {  // fault injection for the kernel's bounds checks
        const int32_t bad_tile = s.n_tiles + 7;
        const size_t i = (size_t)(kn.debug_corrupt_entry - 1) % s.tile_list.size();
        PL_CK(cudaMemcpy(pl->d_tiles + i, &bad_tile, sizeof(int32_t), cudaMemcpyHostToDevice));
    }
    if (!s.transfers.empty())
        PL_CK(cudaMemcpy(pl->d_transfers, s.transfers.data(), s.transfers.size() * sizeof(int32_t),
                         cudaMemcpyHostToDevice));
    if (kn.debug_corrupt_entry > 0 && !s.transfers.empty()) {  // (the host keeps its own valid copy)
        const int32_t bad_code = (int32_t)n_flags + 3;
        const size_t i = (size_t)(kn.debug_corrupt_entry - 1) % s.transfers.size();
        PL_CK(cudaMemcpy(pl->d_transfers + i, &bad_code, sizeof(int32_t), cudaMemcpyHostToDevice));
    }
    PL_CK(cudaMemset(pl->d_err, 0, 4 * sizeof(int32_t)));
    PL_CK(cudaMemset(pl->d_in_flags, 0, n_flags * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_in_cnt, 0, 2 * n_flags * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_out_flags, 0, (size_t)s.n_rc * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_out_cnt, 0, 2 * (size_t)s.n_rc * sizeof(uint32_t)));
    PL_CK(cudaMemset(pl->d_stats, 0, 2 * sizeof(unsigned long long)));
    if (kn.trace >= 2) {
        PL_CK(cudaMalloc(&pl->d_trace, 5 * (size_t)s.n_tiles * sizeof(unsigned long long)));
        PL_CK(cudaMemset(pl->d_trace, 0, 5 * (size_t)s.n_tiles * sizeof(unsigned long long)));
    }
    if (pl->lc.red) {
        // GEMM-RS: the local block's partial rows, stored by the epilogue for
        // the reducer warps; GEMM-AR: the peer sums S, stored by the reducer
        // warps for the epilogue
        pl->red_bytes = (size_t)(s.op == SYN_OP_GEMM_RS ? s.M_r : s.M) * s.N * sizeof(float);
        PL_CK(cudaMalloc(&pl->d_red, pl->red_bytes));
    }
    if (push_ded) {
        for (int rc = 0; rc < s.n_rc; ++rc)
            if ((chunk_row0(s.rb, rc + 1) - chunk_row0(s.rb, rc)) % 32 != 0)
                return bail(SYN_ERR_UNSUPPORTED, "push_sms needs chunks of a multiple of 32 rows");
        // the send row chunks (every chunk of another rank's block), in the
        // order the tile walk produces them: destinations in ring order
        // r + 1, r + 2, ..., then chunk index
        std::vector<int32_t> lst;
        for (int d = 1; d < s.R; ++d) {
            const int q = (s.rank + d) % s.R;
            for (int j = 0; j < s.split; ++j) lst.push_back(q * s.split + j);
        }
        pl->n_push = (int)lst.size();
        PL_CK(cudaMalloc(&pl->d_push, (size_t)s.M * s.N * sizeof(float)));
        PL_CK(cudaMalloc(&pl->d_push_list, std::max<size_t>(1, lst.size()) * sizeof(int32_t)));
        if (!lst.empty())
            PL_CK(cudaMemcpy(pl->d_push_list, lst.data(), lst.size() * sizeof(int32_t), cudaMemcpyHostToDevice));
    }
    if (staged_peers(pl)) {
        pl->recv_slot_rows = (s.op == SYN_OP_GEMM_RS) ? s.M_r : s.M;
        pl->recv_bytes = (uint64_t)(s.R - 1) * pl->recv_slot_rows * s.N * sizeof(float);
        if (pl->recv_bytes > 0) PL_CK(cudaMalloc(&pl->d_recv, pl->recv_bytes));
    }
    PL_CK(cudaStreamCreateWithFlags(&pl->side, cudaStreamNonBlocking));
    if (kn.backend == SYN_BACKEND_CE) {
        const int n = kn.ce_streams > 0 ? std::min(kn.ce_streams, 16) : 4;
        pl->ce_side.push_back(pl->side);
        for (int i = 1; i < n; ++i) {
            cudaStream_t x = nullptr;
            PL_CK(cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking));
            pl->ce_side.push_back(x);
        }
        for (int i = 0; i < n; ++i) {
            cudaEvent_t e = nullptr;
            PL_CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
            pl->ce_join.push_back(e);
        }
    }
    PL_CK(cudaEventCreateWithFlags(&pl->ev_fork, cudaEventDisableTiming));
    PL_CK(cudaEventCreateWithFlags(&pl->ev_join, cudaEventDisableTiming));
    if (kn.backend == SYN_BACKEND_DECOMPOSED) {
        pl->ev_transfer.resize(s.transfers.size(), nullptr);
        for (auto &e : pl->ev_transfer) PL_CK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        // contiguous tile-list ranges with equal arrival key: one launch each
        int t0 = 0;
        for (int t = 1; t <= s.n_tiles; ++t) {
            if (t == s.n_tiles || s.tile_key[t] != s.tile_key[t0]) {
                pl->groups.emplace_back(t0, t);
                pl->group_key.push_back(s.tile_key[t0]);
                t0 = t;
            }
        }
    }
    PL_CK(cudaDeviceSynchronize());
#undef PL_CK
    *out = pl;
    return SYN_OK;
}

// A2A-GEMM row blocks: validated counts and their sum.
int a2a_rows(int R, const int64_t *rows_from, int64_t &M) {
    if (rows_from == nullptr) return fail(SYN_ERR_INVALID, "null rows_from");
    if (R < 1) return fail(SYN_ERR_INVALID, "R must be >= 1");
    if (R > kMaxRanks) return fail(SYN_ERR_UNSUPPORTED, "R > 8");
    M = 0;
    for (int q = 0; q < R; ++q) {
        if (rows_from[q] < 0) return fail(SYN_ERR_INVALID, "rows_from entries must be >= 0");
        M += rows_from[q];
    }
    if (M == 0) return fail(SYN_ERR_INVALID, "no rows to multiply (every rows_from entry is 0)");
    return SYN_OK;
}

}  // namespace

extern "C" {

int syn_plan_create(syn_plan_t *out, syn_op_t op, int R, int rank, const syn_layout_t *layout,
                    int64_t chunk_rows, int split, syn_order_t order, const syn_knobs_t *knobs) {
    return plan_create(out, op, R, rank, layout, chunk_rows, split, order, knobs, nullptr);
}

int syn_plan_create_a2a(syn_plan_t *out, int R, int rank, const int64_t *rows_from, int64_t N, int64_t K,
                        int split, syn_order_t order, const syn_knobs_t *knobs) {
    if (out == nullptr) return fail(SYN_ERR_INVALID, "null argument");
    *out = nullptr;
    int64_t M = 0;
    int rc = a2a_rows(R, rows_from, M);
    if (rc != SYN_OK) return rc;
    const syn_layout_t L = {M, N, K, 0, 0, 0};
    return plan_create(out, SYN_OP_AG_GEMM, R, rank, &L, 0, split, order, knobs, rows_from);
}

int syn_schedule_build_a2a(int R, int rank, const int64_t *rows_from, int64_t N, int64_t K, int split,
                           syn_order_t order, const syn_knobs_t *knobs, syn_plan_info_t *info,
                           int32_t *tile_list, int32_t *tile_key, int32_t *transfers) {
    int64_t M = 0;
    int rc = a2a_rows(R, rows_from, M);
    if (rc != SYN_OK) return rc;
    const syn_knobs_t kn = resolve_knobs(knobs);
    const syn_layout_t L = {M, N, K, 0, 0, 0};
    Schedule s;
    std::string err;
    rc = build_schedule(SYN_OP_AG_GEMM, R, rank, L, 0, split, order, kn, s, err, rows_from);
    if (rc != SYN_OK) return fail(rc, err);
    if (info) fill_info(s, kn, info);
    if (tile_list) std::memcpy(tile_list, s.tile_list.data(), s.tile_list.size() * sizeof(int32_t));
    if (tile_key) std::memcpy(tile_key, s.tile_key.data(), s.tile_key.size() * sizeof(int32_t));
    if (transfers) std::memcpy(transfers, s.transfers.data(), s.transfers.size() * sizeof(int32_t));
    return SYN_OK;
}

int syn_plan_destroy(syn_plan_t plan) {
    free_plan(plan);
    return SYN_OK;
}

}  // extern "C"

namespace {

// AG-GEMM and A2A-GEMM: source q's rows go to rows [off[q], off[q+1]) of
// `gathered`, then C = gathered . B.
int gather_gemm(syn_plan_t plan, bool a2a, const void *const *shards, void *gathered, const void *B, void *C,
                void *stream) {
    int rc = check_plan(plan, SYN_OP_AG_GEMM, a2a);
    if (rc != SYN_OK) return rc;
    if (shards == nullptr || gathered == nullptr || B == nullptr || C == nullptr)
        return fail(SYN_ERR_INVALID, "null operand");
    const Schedule &s = plan->s;
    for (int q = 0; q < s.R; ++q)
        if ((shards[q] == nullptr && block_rows(s.rb, q) > 0) || !aligned16(shards[q]))
            return fail(SYN_ERR_INVALID, "shard pointer null or not 16-byte aligned");
    if (!aligned16(gathered) || !aligned16(B) || !aligned16(C))
        return fail(SYN_ERR_INVALID, "operand not 16-byte aligned");
    const int64_t row_bytes = s.K * 2;
    // tensor maps (cached on the operand pointers)
    const bool direct = plan->kn.direct_fetch != 0;
    std::vector<const void *> key = {gathered, B, C};
    if (direct)
        for (int q = 0; q < s.R; ++q) key.push_back(shards[q]);
    if (key != plan->map_key) {
        if ((rc = encode_operands(plan, gathered, B)) != SYN_OK) return rc;
        // bf16 tile stores of the epilogue: 32 columns x 32 rows, 64-byte swizzle
        if ((rc = encode_2d(&plan->maps.c, C, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.N, s.M, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_64B)) != SYN_OK)
            return rc;
        // direct fetch: each source shard as an A operand in place (same boxes as `gathered`)
        if (direct) {
            const int tk = plan->lc.tile_k;
            const CUtensorMapSwizzle a_swz = tk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
            for (int q = 0; q < s.R; ++q) {
                const int64_t rows = block_rows(s.rb, q);
                if (rows == 0) continue;
                if ((rc = encode_2d(&plan->maps.peer[q], shards[q], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.K,
                                    (uint64_t)rows, tk, 128, a_swz)) != SYN_OK)
                    return rc;
            }
        }
        plan->map_key = key;
    }
    plan->epoch += 1;
    KernelParams p = base_params(plan);
    for (int q = 0; q < s.R; ++q) p.stage_src[q] = static_cast<const uint8_t *>(shards[q]);
    p.stage_dst = static_cast<uint8_t *>(gathered);
    p.row_bytes = row_bytes;
    p.local_inplace =
        (static_cast<const uint8_t *>(shards[s.rank]) ==
         static_cast<uint8_t *>(gathered) + s.rb.off[s.rank] * row_bytes)
            ? 1
            : 0;
    p.out = static_cast<uint16_t *>(C);
    p.f32_out = nullptr;
    p.epi_tma = 1;
    p.direct_fetch = direct ? 1 : 0;  // (only where the backend's tiles wait on flags)
    return run(plan, p, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int syn_ag_gemm(syn_plan_t plan, const void *const *shards, void *gathered, const void *B, void *C,
                void *stream) {
    return gather_gemm(plan, false, shards, gathered, B, C, stream);
}

int syn_a2a_gemm(syn_plan_t plan, const void *const *parts, void *gathered, const void *B, void *C,
                 void *stream) {
    return gather_gemm(plan, true, parts, gathered, B, C, stream);
}

static int rs_ar_call(syn_plan_t plan, int op, const void *A, const void *B,
                      const float *const *peers, float *f32_out, void *out, void *stream) {
    int rc = check_plan(plan, op);
    if (rc != SYN_OK) return rc;
    if (A == nullptr || B == nullptr || peers == nullptr || out == nullptr)
        return fail(SYN_ERR_INVALID, "null operand");
    const Schedule &s = plan->s;
    for (int q = 0; q < s.R; ++q)
        if (q != s.rank && (peers[q] == nullptr || !aligned16(peers[q])))
            return fail(SYN_ERR_INVALID, "peer partial null or not 16-byte aligned");
    if (!aligned16(A) || !aligned16(B) || !aligned16(out) || (f32_out && !aligned16(f32_out)))
        return fail(SYN_ERR_INVALID, "operand not 16-byte aligned");
    const bool staged = staged_peers(plan);
    // reducer warps: where the epilogue leaves the reducing tiles' fp32 partials
    float *red_buf = nullptr;
    int64_t red_rows = 0;
    int32_t red_row_off = 0;
    if (plan->lc.red) {
        red_buf = plan->d_red;
        if (op == SYN_OP_GEMM_RS) {
            red_rows = s.M_r;
            red_row_off = (int32_t)(s.rank * s.M_r);
        } else {
            red_rows = s.M;
        }
    }
    std::vector<const void *> key = {A, B, f32_out, red_buf, out};
    if (!staged)
        for (int q = 0; q < s.R; ++q) key.push_back(q == s.rank ? nullptr : peers[q]);
    if (key != plan->map_key) {
        if ((rc = encode_operands(plan, A, B)) != SYN_OK) return rc;
        for (int q = 0; q < s.R; ++q) {
            if (q == s.rank) continue;
            const void *base;
            uint64_t rows;
            if (staged) {
                base = plan->d_recv + (uint64_t)recv_slot(q, s.rank) * plan->recv_slot_rows * s.N * 4;
                rows = (uint64_t)plan->recv_slot_rows;
            } else {
                base = peers[q];
                rows = (uint64_t)s.M;
            }
            if ((rc = encode_2d(&plan->maps.peer[q], base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.N, rows,
                                32, 128)) != SYN_OK)
                return rc;
        }
        // fp32 tile stores of the epilogue (used by instances with staging room):
        // 32 columns x 32 rows, 128-byte swizzle; with dedicated push CTAs the
        // send rows go to the plan's push buffer first
        const bool push_ded = op == SYN_OP_GEMM_RS && plan->d_push != nullptr && f32_out != nullptr;
        if (f32_out != nullptr &&
            (rc = encode_2d(&plan->maps.f32out, push_ded ? plan->d_push : f32_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                            4, s.N, s.M, 32, 32)) != SYN_OK)
            return rc;
        // the push CTAs' boxes: 256 columns x 32 rows, no swizzle
        if (push_ded &&
            ((rc = encode_2d(&plan->maps.push_src, plan->d_push, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.N, s.M,
                             kPushBoxCols, 32, CU_TENSOR_MAP_SWIZZLE_NONE)) != SYN_OK ||
             (rc = encode_2d(&plan->maps.push_dst, f32_out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.N, s.M,
                             kPushBoxCols, 32, CU_TENSOR_MAP_SWIZZLE_NONE)) != SYN_OK))
            return rc;
        if (red_buf != nullptr &&
            (rc = encode_2d(&plan->maps.red, red_buf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.N,
                            (uint64_t)red_rows, 32, 32)) != SYN_OK)
            return rc;
        // GEMM-AR with reducer warps: bf16 tile stores of out by the epilogue,
        // 32 columns x 32 rows, 64-byte swizzle
        if (op == SYN_OP_GEMM_AR && plan->lc.red &&
            (rc = encode_2d(&plan->maps.c, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.N, s.M, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_64B)) != SYN_OK)
            return rc;
        plan->map_key = key;
    }
    plan->epoch += 1;
    KernelParams p = base_params(plan);
    for (int q = 0; q < s.R; ++q)
        p.stage_src[q] = q == s.rank ? nullptr : reinterpret_cast<const uint8_t *>(peers[q]);
    p.stage_dst = plan->d_recv;
    p.row_bytes = s.N * 4;
    p.red_buf = red_buf;
    p.red_row_off = red_row_off;
    p.epi_tma = 1;
    p.send_push = (op == SYN_OP_GEMM_RS && plan->kn.rs_push) ? 1 : 0;
    if (p.send_push && plan->d_push != nullptr && f32_out != nullptr) {
        // dedicated push CTAs add the produced rows; the epilogue only stores them
        p.send_push = 0;
        p.push_dedicated = 1;
        p.push_buf = plan->d_push;
        p.push_list = plan->d_push_list;
        p.n_push = plan->n_push;
    }
    p.recv_slot_rows = plan->recv_slot_rows;
    p.peer_row_off = (staged && op == SYN_OP_GEMM_RS) ? (int32_t)(s.rank * s.M_r) : 0;
    p.out = static_cast<uint16_t *>(out);
    p.f32_out = f32_out;
    return run(plan, p, static_cast<cudaStream_t>(stream));
}

int syn_gemm_rs(syn_plan_t plan, const void *A, const void *B, const float *const *peer_partials,
                float *send, void *out_r, void *stream) {
    return rs_ar_call(plan, SYN_OP_GEMM_RS, A, B, peer_partials, send, out_r, stream);
}

int syn_gemm_ar(syn_plan_t plan, const void *A, const void *B, const float *const *peer_partials,
                float *publish, void *out, void *stream) {
    return rs_ar_call(plan, SYN_OP_GEMM_AR, A, B, peer_partials, publish, out, stream);
}

int syn_sync_status(syn_plan_t plan, void *stream) {
    if (plan == nullptr) return fail(SYN_ERR_INVALID, "null plan");
    SYN_CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    SYN_CK(cudaStreamSynchronize(plan->side));
    for (cudaStream_t x : plan->ce_side) SYN_CK(cudaStreamSynchronize(x));
    int32_t e[4] = {0, 0, 0, 0};
    SYN_CK(cudaMemcpy(e, plan->d_err, sizeof(e), cudaMemcpyDeviceToHost));
    if (e[0] == 0) return SYN_OK;
    const size_t n_flags = (size_t)plan->s.n_rc * plan->s.R;
    SYN_CK(cudaMemset(plan->d_err, 0, 4 * sizeof(int32_t)));
    SYN_CK(cudaMemset(plan->d_in_cnt, 0, 2 * n_flags * sizeof(uint32_t)));
    SYN_CK(cudaMemset(plan->d_out_cnt, 0, 2 * (size_t)plan->s.n_rc * sizeof(uint32_t)));
    SYN_CK(cudaDeviceSynchronize());
    return fail(e[0], std::string("device error ") + syn_status_string(e[0]) + " at site " +
                          std::to_string(e[1]) + " in CTA " + std::to_string(e[2]) + " (info " +
                          std::to_string(e[3]) + ")");
}

int syn_plan_query(syn_plan_t plan, syn_plan_info_t *info) {
    if (plan == nullptr || info == nullptr) return fail(SYN_ERR_INVALID, "null argument");
    fill_info(plan->s, plan->kn, info);
    info->grid_compute = plan->grid_compute;
    info->grid_comm = plan->grid_comm;
    info->smem_bytes = plan->smem;
    info->num_sms = plan->num_sms;
    info->epoch = plan->epoch;
    info->recv_bytes = plan->recv_bytes;
    return SYN_OK;
}

int syn_plan_tables(syn_plan_t plan, int32_t *tile_list, int32_t *tile_key, int32_t *transfers) {
    if (plan == nullptr) return fail(SYN_ERR_INVALID, "null plan");
    const Schedule &s = plan->s;
    if (tile_list) std::memcpy(tile_list, s.tile_list.data(), s.tile_list.size() * sizeof(int32_t));
    if (tile_key) std::memcpy(tile_key, s.tile_key.data(), s.tile_key.size() * sizeof(int32_t));
    if (transfers) std::memcpy(transfers, s.transfers.data(), s.transfers.size() * sizeof(int32_t));
    return SYN_OK;
}

int syn_plan_flags(syn_plan_t plan, uint32_t *in_flags, uint32_t *out_flags) {
    if (plan == nullptr) return fail(SYN_ERR_INVALID, "null plan");
    SYN_CK(cudaDeviceSynchronize());
    if (in_flags)
        SYN_CK(cudaMemcpy(in_flags, plan->d_in_flags, (size_t)plan->s.n_rc * plan->s.R * sizeof(uint32_t),
                          cudaMemcpyDeviceToHost));
    if (out_flags)
        SYN_CK(cudaMemcpy(out_flags, plan->d_out_flags, (size_t)plan->s.n_rc * sizeof(uint32_t),
                          cudaMemcpyDeviceToHost));
    return SYN_OK;
}

int syn_plan_trace(syn_plan_t plan, uint64_t *out) {
    if (plan == nullptr || out == nullptr) return fail(SYN_ERR_INVALID, "null argument");
    if (plan->d_trace == nullptr) return fail(SYN_ERR_INVALID, "plan was created without trace = 2");
    SYN_CK(cudaDeviceSynchronize());
    SYN_CK(cudaMemcpy(out, plan->d_trace, 5 * (size_t)plan->s.n_tiles * sizeof(uint64_t),
                      cudaMemcpyDeviceToHost));
    return SYN_OK;
}

int syn_plan_stats(syn_plan_t plan, uint64_t *flag_wait_ns, uint64_t *cta_busy_ns) {
    if (plan == nullptr) return fail(SYN_ERR_INVALID, "null plan");
    unsigned long long v[2] = {0, 0};
    SYN_CK(cudaDeviceSynchronize());
    SYN_CK(cudaMemcpy(v, plan->d_stats, sizeof(v), cudaMemcpyDeviceToHost));
    if (flag_wait_ns) *flag_wait_ns = v[0];
    if (cta_busy_ns) *cta_busy_ns = v[1];
    return SYN_OK;
}

const char *syn_status_string(int status) {
    switch (status) {
        case SYN_OK: return "SYN_OK";
        case SYN_ERR_INVALID: return "SYN_ERR_INVALID";
        case SYN_ERR_UNSUPPORTED: return "SYN_ERR_UNSUPPORTED";
        case SYN_ERR_CUDA: return "SYN_ERR_CUDA";
        case SYN_ERR_TIMEOUT: return "SYN_ERR_TIMEOUT";
        case SYN_ERR_BOUNDS: return "SYN_ERR_BOUNDS";
        default: return "SYN_ERR_UNKNOWN";
    }
}

const char *syn_last_error(void) { return g_err.c_str(); }

}  // extern "C"
