// noalloc.cu -- AG-GEMM entry point that allocates no device memory.
//
// Why it exists: some callers cannot allocate device memory themselves or let
// a library do it.  Plug-in hosts (inference-server backends, framework custom
// ops running under a caching allocator) hand an operator only its input and
// output tensors and own every allocation; latency-bound serving loops forbid
// cudaMalloc / cudaFree after start-up because those calls can synchronise the
// whole device and can fail mid-step.  syn_plan_create allocates the plan's
// flags, counters and tables with cudaMalloc, so those callers cannot use it.
//
// This variant keeps that scratch in one file-scope __device__ array of fixed,
// modest size (SYN_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the
// library until the process exits) and runs the same fused AG-GEMM kernel with
// the co-located TMA staging backend, so the whole call is two kernel
// launches: a small one that fills that array, then the GEMM.  The caller
// passes inputs and outputs.
//
// Host code never dereferences or passes the array's name to a kernel: in host
// code that name is only a stand-in for the symbol.  The device address is
// looked up once per device with cudaGetSymbolAddress (with that device
// current) during the first call on that device.
//
// Each call writes its tile and transfer lists into the array, and clears the
// flags, counters and error word, with one small kernel that receives the
// lists by value as its parameter block (at most 16.6 KB): no host buffer
// has to outlive the call, and nothing waits for the host.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>
#include <string>

#include "fused.h"
#include "host_util.h"
#include "schedule.h"
#include "syn.h"

using namespace syn;

namespace {

// Layout of the scratch array (byte offsets).
constexpr int kOffTiles = 0;
constexpr int kOffTransfers = kOffTiles + SYN_NOALLOC_MAX_TILES * 4;
constexpr int kMaxFlags = SYN_NOALLOC_MAX_ROW_CHUNKS * kMaxRanks;
constexpr int kOffInFlags = kOffTransfers + SYN_NOALLOC_MAX_ROW_CHUNKS * 4;
constexpr int kOffInCnt = kOffInFlags + kMaxFlags * 4;
constexpr int kOffOutFlags = kOffInCnt + 2 * kMaxFlags * 4;
constexpr int kOffOutCnt = kOffOutFlags + SYN_NOALLOC_MAX_ROW_CHUNKS * 4;
constexpr int kOffErr = kOffOutCnt + 2 * SYN_NOALLOC_MAX_ROW_CHUNKS * 4;
constexpr int kUsed = kOffErr + 4 * 4;
static_assert(kUsed <= SYN_NOALLOC_SCRATCH_BYTES, "scratch layout exceeds the declared size");

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

int fail(int code, const std::string &msg) {
    syn::set_last_error(msg);
    return code;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool encode(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
            uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The scratch: tile list, transfer list, ready flags, slice and producer
// counters and the error word of the call in flight.
static __device__ __align__(256) unsigned char g_syn_noalloc_scratch[SYN_NOALLOC_SCRATCH_BYTES];

namespace {

// One call's schedule tables, passed by value to the fill kernel.
struct NoallocTables {
    int32_t n_tiles, n_transfers;
    int32_t tiles[SYN_NOALLOC_MAX_TILES];
    int32_t transfers[SYN_NOALLOC_MAX_ROW_CHUNKS];
};
static_assert(sizeof(NoallocTables) <= 32000, "kernel parameter block limit");

// Writes the tables into the scratch array and zeroes everything after them
// (flags, counters, error word).  Device code names the array directly.
__global__ void noalloc_fill(const __grid_constant__ NoallocTables t) {
    int32_t *tiles = reinterpret_cast<int32_t *>(g_syn_noalloc_scratch + kOffTiles);
    int32_t *transfers = reinterpret_cast<int32_t *>(g_syn_noalloc_scratch + kOffTransfers);
    uint32_t *clear = reinterpret_cast<uint32_t *>(g_syn_noalloc_scratch + kOffInFlags);
    constexpr int n_clear = (kUsed - kOffInFlags) / 4;
    const int stride = (int)(gridDim.x * blockDim.x);
    for (int i = (int)(blockIdx.x * blockDim.x + threadIdx.x); i < SYN_NOALLOC_MAX_TILES; i += stride) {
        if (i < t.n_tiles) tiles[i] = t.tiles[i];
        if (i < t.n_transfers && i < SYN_NOALLOC_MAX_ROW_CHUNKS) transfers[i] = t.transfers[i];
        if (i < n_clear) clear[i] = 0u;
    }
}
static_assert((kUsed - kOffInFlags) / 4 <= SYN_NOALLOC_MAX_TILES, "one pass of the fill loop clears the rest");
static_assert(kOffInFlags % 4 == 0 && kUsed % 4 == 0, "word-aligned layout");

}  // namespace

extern "C" int syn_ag_gemm_noalloc(int R, int rank, const syn_layout_t *layout, int split,
                                   syn_order_t order, const void *const *shards, void *gathered,
                                   const void *B, void *C, int32_t *status_dev, void *stream) {
    if (layout == nullptr || shards == nullptr || gathered == nullptr || B == nullptr || C == nullptr)
        return fail(SYN_ERR_INVALID, "null argument");
    syn_knobs_t kn;
    syn_knobs_default(&kn);
    kn.backend = SYN_BACKEND_TMA_COLOCATED;
    kn.tile_n = (layout->N % 256 == 0) ? 256 : 128;
    kn.timeout_ns = syn::host_timeout_ns();  // as plans: SYN_TIMEOUT_NS, else 2 s
    Schedule s;
    std::string err;
    int rc = build_schedule(SYN_OP_AG_GEMM, R, rank, *layout, 0, split, order, kn, s, err);
    if (rc != SYN_OK) return fail(rc, err);
    if (s.n_tiles > SYN_NOALLOC_MAX_TILES)
        return fail(SYN_ERR_UNSUPPORTED, "syn_ag_gemm_noalloc: " + std::to_string(s.n_tiles) +
                                             " output tiles exceed SYN_NOALLOC_MAX_TILES (" +
                                             std::to_string(SYN_NOALLOC_MAX_TILES) + ")");
    if (s.n_rc > SYN_NOALLOC_MAX_ROW_CHUNKS)
        return fail(SYN_ERR_UNSUPPORTED, "syn_ag_gemm_noalloc: " + std::to_string(s.n_rc) +
                                             " chunks exceed SYN_NOALLOC_MAX_ROW_CHUNKS (" +
                                             std::to_string(SYN_NOALLOC_MAX_ROW_CHUNKS) + ")");
    for (int q = 0; q < R; ++q)
        if (shards[q] == nullptr || (reinterpret_cast<uintptr_t>(shards[q]) & 15u))
            return fail(SYN_ERR_INVALID, "shard pointer null or not 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(gathered) | reinterpret_cast<uintptr_t>(B) |
         reinterpret_cast<uintptr_t>(C)) & 15u)
        return fail(SYN_ERR_INVALID, "operand not 16-byte aligned");

    // ---- set-up, once per device: the scratch array's device address ----
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(SYN_ERR_CUDA, "cudaGetDevice failed or device index out of range");
    uint8_t *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_scratch_addr[dev] == nullptr) {
            void *ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_syn_noalloc_scratch);
            if (e != cudaSuccess || ptr == nullptr)
                return fail(SYN_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            g_scratch_addr[dev] = ptr;
        }
        scratch = static_cast<uint8_t *>(g_scratch_addr[dev]);
    }
    int num_sms = 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(SYN_ERR_CUDA, "cudaDeviceGetAttribute failed");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // ---- this call's tables in, flags / counters / error word cleared ----
    // (the array keeps the previous call's contents)
    if (s.transfers.size() > (size_t)SYN_NOALLOC_MAX_ROW_CHUNKS)
        return fail(SYN_ERR_UNSUPPORTED, "syn_ag_gemm_noalloc: too many staging transfers");
    {
        NoallocTables t;
        std::memset(&t, 0, sizeof(t));
        t.n_tiles = s.n_tiles;
        t.n_transfers = (int32_t)s.transfers.size();
        std::memcpy(t.tiles, s.tile_list.data(), s.tile_list.size() * 4);
        std::memcpy(t.transfers, s.transfers.data(), s.transfers.size() * 4);
        noalloc_fill<<<8, 256, 0, st>>>(t);
        const cudaError_t fe = cudaGetLastError();
        if (fe != cudaSuccess)
            return fail(SYN_ERR_CUDA, std::string("writing the schedule into the scratch array: ") +
                                          cudaGetErrorString(fe));
    }

    TensorMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    if (!encode(&maps.a, gathered, (uint64_t)s.K, (uint64_t)s.M, 64, 128) ||
        !encode(&maps.b, B, (uint64_t)s.N, (uint64_t)s.K, 64, 64))
        return fail(SYN_ERR_CUDA, "cuTensorMapEncodeTiled failed");

    KernelParams p;
    std::memset(&p, 0, sizeof(p));
    p.op = OP_AG;
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
    p.G = s.n_tiles < num_sms ? s.n_tiles : num_sms;
    p.colocated = 1;
    p.waits = 1;
    p.drop_transfer = -1;
    p.delay_transfer = -1;
    p.epoch = 1;  // flags were cleared, so every call can use the same epoch
    p.timeout_ns = kn.timeout_ns;
    p.tile_list = reinterpret_cast<const int32_t *>(scratch + kOffTiles);
    p.transfers = reinterpret_cast<const int32_t *>(scratch + kOffTransfers);
    p.n_transfers = (int32_t)s.transfers.size();
    p.in_flags = reinterpret_cast<uint32_t *>(scratch + kOffInFlags);
    p.in_cnt = reinterpret_cast<uint32_t *>(scratch + kOffInCnt);
    p.out_flags = reinterpret_cast<uint32_t *>(scratch + kOffOutFlags);
    p.out_cnt = reinterpret_cast<uint32_t *>(scratch + kOffOutCnt);
    p.err = reinterpret_cast<int32_t *>(scratch + kOffErr);
    p.stats = nullptr;
    for (int q = 0; q < s.R; ++q) p.stage_src[q] = static_cast<const uint8_t *>(shards[q]);
    p.stage_dst = static_cast<uint8_t *>(gathered);
    p.row_bytes = s.K * 2;
    p.local_inplace = (static_cast<const uint8_t *>(shards[s.rank]) ==
                       static_cast<uint8_t *>(gathered) + (int64_t)s.rank * s.M_r * s.K * 2)
                          ? 1
                          : 0;
    const int64_t tbytes = (int64_t)p.cr * p.row_bytes;
    int64_t slice = 128 * 1024;
    if (slice > tbytes) slice = tbytes;
    p.slice_bytes = (int32_t)slice;
    p.slices_per_transfer = (int32_t)((tbytes + slice - 1) / slice);
    p.out = static_cast<uint16_t *>(C);
    p.f32_out = nullptr;

    LaunchCfg lc;
    lc.tile_n = s.tile_n;
    lc.tile_k = 64;
    lc.stg = true;
    lc.pair = false;
    lc.stages = default_stages(OP_AG, s.tile_n, lc.tile_k, lc.stg, lc.pair);
    lc.grid = p.G;
    const cudaError_t le = launch_fused_ag(p, maps, lc, st);
    if (le != cudaSuccess) return fail(SYN_ERR_CUDA, std::string("launch: ") + cudaGetErrorString(le));
    if (status_dev != nullptr &&
        cudaMemcpyAsync(status_dev, scratch + kOffErr, 4 * sizeof(int32_t), cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
        return fail(SYN_ERR_CUDA, "copying the device status out failed");
    return SYN_OK;
}
