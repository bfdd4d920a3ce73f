// api.cu -- the extern "C" entry points of libfp8bq: argument checks, the
// per-shape variant table, the device status word, and the launches.
#include <dlfcn.h>

#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <tuple>

#include "internal.h"

namespace fp8bq {

// ------------------------------------------------------- device state

// Status word the kernels' bounded waits write on time-out.
__device__ int g_status_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int ready = 0;
    int supported = 0;
    int num_sms = 0;
    int* status = nullptr;  // device address of g_status_word
    std::string name;       // spaces replaced by '_'
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

fp8bq_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8BQ_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FP8BQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
            cudaGetLastError();
            return FP8BQ_ERR_CUDA;
        }
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return FP8BQ_ERR_CUDA;
        }
        d.status = static_cast<int*>(p);
        d.num_sms = prop.multiProcessorCount;
        d.supported = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
        d.name = prop.name;
        for (char& c : d.name)
            if (c == ' ') c = '_';
        d.ready = 1;
    }
    *out = &d;
    return d.supported ? FP8BQ_OK : FP8BQ_ERR_UNSUPPORTED;
}

uint64_t wait_timeout_ns() {
    static uint64_t ns = [] {
        const char* e = std::getenv("FP8BQ_WAIT_TIMEOUT_MS");
        double ms = e ? std::atof(e) : 2000.0;
        if (!(ms > 0.0)) ms = 2000.0;
        return static_cast<uint64_t>(ms * 1e6);
    }();
    return ns;
}

fp8bq_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FP8BQ_OK;
    cudaGetLastError();  // clear the non-sticky error state for the next call
    log_error(cudaGetErrorString(e));
    return FP8BQ_ERR_LAUNCH;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// ------------------------------------------------------- variant table
//
// Text file, one entry per line:  N K fmt out M kind block_n split grid [mma_scale]
// (fmt: fp32|ue8m0, or a table-only format below; out: bf16|fp16|fp32; kind:
// normal|swap|swap64; mma_scale 0 when absent).  Per
// (N, K, fmt, out) the entries form an M grid; a lookup takes the grid point
// nearest to M, the smaller one on a tie ("vLLM 量化 Kernel 配置机制" §4.2:
// the key with the least |key - M|, e.g. M=37 -> 32, M=2050 -> 2048).

using TableKey = std::tuple<int64_t, int64_t, int, int>;  // N, K, fmt, out

struct Table {
    bool loaded = false;
    std::string path;
    std::map<TableKey, std::map<int64_t, fp8bq_variant>> rows;
    std::set<TableKey> logged;
};

std::mutex g_table_mutex;
Table g_table;

std::string library_dir() {
    Dl_info info;
    if (dladdr(reinterpret_cast<void*>(&library_dir), &info) && info.dli_fname) {
        std::string p = info.dli_fname;
        size_t cut = p.find_last_of('/');
        if (cut != std::string::npos) return p.substr(0, cut);
    }
    return ".";
}

std::string table_path(const std::string& device_name) {
    const char* e = std::getenv("FP8BQ_TABLE");
    if (e && *e) return e;
    if (device_name.empty()) return std::string();
    return library_dir() + "/../tables/" + device_name + ".tbl";
}

// Table-only format codes of the other GEMMs, each with its own measured
// shapes: rowwise e4m3 (FP8_Dynamic) "rw8", rowwise INT8 "ri8", block INT8
// "bi8" (for INT8, mma_scale 1 = the two-plane kernel), and the grouped (MoE)
// GEMM with fp32 or UE8M0 scales, "gfp32" / "gue8m0" (M = rows per expert).
constexpr int kTableRowwiseE4m3 = 2;
constexpr int kTableRowwiseInt8 = 3;
constexpr int kTableBlockInt8 = 4;
constexpr int kTableGroupedFp32 = 5;
constexpr int kTableGroupedUe8m0 = 6;

int parse_fmt(const char* s) {
    if (!std::strcmp(s, "fp32")) return FP8BQ_SCALE_FP32;
    if (!std::strcmp(s, "ue8m0")) return FP8BQ_SCALE_UE8M0;
    if (!std::strcmp(s, "rw8")) return kTableRowwiseE4m3;
    if (!std::strcmp(s, "ri8")) return kTableRowwiseInt8;
    if (!std::strcmp(s, "bi8")) return kTableBlockInt8;
    if (!std::strcmp(s, "gfp32")) return kTableGroupedFp32;
    if (!std::strcmp(s, "gue8m0")) return kTableGroupedUe8m0;
    return -1;
}
int parse_out(const char* s) {
    if (!std::strcmp(s, "bf16")) return FP8BQ_BF16;
    if (!std::strcmp(s, "fp16")) return FP8BQ_FP16;
    if (!std::strcmp(s, "fp32")) return FP8BQ_FP32;
    return -1;
}
int parse_kind(const char* s) {
    if (!std::strcmp(s, "normal")) return FP8BQ_KIND_NORMAL;
    if (!std::strcmp(s, "swap")) return FP8BQ_KIND_SWAP_AB;
    if (!std::strcmp(s, "swap64")) return FP8BQ_KIND_SWAP_AB_64;
    return -1;
}

void load_table_locked(const std::string& device_name) {
    g_table.rows.clear();
    g_table.logged.clear();
    g_table.path = table_path(device_name);
    g_table.loaded = true;
    if (g_table.path.empty()) return;
    FILE* f = std::fopen(g_table.path.c_str(), "r");
    if (!f) return;  // a missing table only costs speed
    char line[512];
    while (std::fgets(line, sizeof line, f)) {
        char* hash = std::strchr(line, '#');
        if (hash) *hash = 0;
        long long N, K, M;
        char fmt[16], out[16], kind[16];
        int bn, split, grid, mma_scale = 0;
        const int got = std::sscanf(line, "%lld %lld %15s %15s %lld %15s %d %d %d %d", &N, &K, fmt,
                                    out, &M, kind, &bn, &split, &grid, &mma_scale);
        if (got != 9 && got != 10) continue;  // blank or malformed line: skipped
        const int ifmt = parse_fmt(fmt), iout = parse_out(out), ikind = parse_kind(kind);
        if (ifmt < 0 || iout < 0 || ikind < 0 || M < 0) continue;
        fp8bq_variant v = {};
        v.kind = ikind;
        v.block_n = bn;
        v.split = split;
        v.grid = grid;
        v.mma_scale = mma_scale;
        v.from_table = 1;
        g_table.rows[TableKey(N, K, ifmt, iout)][M] = v;
    }
    std::fclose(f);
}

// Default variant when the table has no entry (speed only, never correctness;
// "vLLM 量化 Kernel 配置机制" §4.1).  Swap-AB below 129 tokens, otherwise the
// normal orientation with 256-wide weight tiles.  When the tiles cannot keep
// every SM busy for whole waves, the (tile, K-slab) units are shared out
// evenly (stream-K, split = 0); the tile count must fit the workspace's
// counter prefix for that.  With UE8M0 scales and whole groups of four K
// slabs, the tensor core applies the scales (block-scaled MMA) on 128-wide and
// wider tiles, where it measured faster on GB300.
fp8bq_variant default_variant(int64_t M, int64_t N, int64_t K, int fmt, int num_sms) {
    fp8bq_variant v = {};
    int64_t tiles;
    if (M <= 128) {
        v.kind = FP8BQ_KIND_SWAP_AB;
        v.block_n = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
        tiles = ((N + 127) / 128) * ((M + v.block_n - 1) / v.block_n);
    } else {
        v.kind = FP8BQ_KIND_NORMAL;
        v.block_n = N >= 256 ? 256 : 128;
        tiles = ((N + v.block_n - 1) / v.block_n) * ((M + 127) / 128);
    }
    const bool fits_counters = tiles * 8 * 4 <= static_cast<int64_t>(kCounterRegion);
    const bool whole_waves = tiles % num_sms == 0 || tiles >= 4 * static_cast<int64_t>(num_sms);
    v.split = (!whole_waves && fits_counters) ? 0 : 1;
    v.grid = 0;
    v.mma_scale = (fmt == FP8BQ_SCALE_UE8M0 && K % (4 * kGroup) == 0 &&
                   (v.kind == FP8BQ_KIND_NORMAL || v.block_n >= 64))
                      ? 1
                      : 0;
    v.from_table = 0;
    return v;
}

// Nearest-M entry of (N, K, fmt, out) in the table; caller holds the lock.
bool table_lookup_locked(int64_t M, int64_t N, int64_t K, int fmt, int out, fp8bq_variant* v) {
    const TableKey key(N, K, fmt, out);
    auto it = g_table.rows.find(key);
    if (it == g_table.rows.end() || it->second.empty()) return false;
    const fp8bq_variant* best = nullptr;
    int64_t best_d = 0;
    for (const auto& kv : it->second) {  // ascending M: strict '<' keeps the smaller on ties
        const int64_t d = kv.first > M ? kv.first - M : M - kv.first;
        if (!best || d < best_d) {
            best = &kv.second;
            best_d = d;
        }
    }
    *v = *best;
    return true;
}

// The table's entry for one of the table-only formats, if it has the shape.
bool format_table_lookup(int table_fmt, int64_t M, int64_t N, int64_t K, int out,
                         const std::string& device_name, fp8bq_variant* v) {
    std::lock_guard<std::mutex> lock(g_table_mutex);
    if (!g_table.loaded) load_table_locked(device_name);
    return table_lookup_locked(M, N, K, table_fmt, out, v);
}

fp8bq_variant select_variant(int64_t M, int64_t N, int64_t K, int fmt, int out,
                             const std::string& device_name, int num_sms) {
    std::lock_guard<std::mutex> lock(g_table_mutex);
    if (!g_table.loaded) load_table_locked(device_name);
    const TableKey key(N, K, fmt, out);
    fp8bq_variant hit;
    if (table_lookup_locked(M, N, K, fmt, out, &hit)) return hit;
    if (g_table.logged.insert(key).second) {
        const char* e = std::getenv("FP8BQ_LOG");
        if (e && std::atoi(e) == 1)
            std::fprintf(stderr,
                         "fp8bq: no table entry for N=%lld K=%lld fmt=%d out=%d (table %s); "
                         "using the default variant\n",
                         static_cast<long long>(N), static_cast<long long>(K), fmt, out,
                         g_table.path.empty() ? "<none>" : g_table.path.c_str());
    }
    return default_variant(M, N, K, fmt, num_sms);
}

// Grouped problems: the tile grid counts every expert as full (the counts
// are on the device).  Token tile from the rows per expert as for a plain
// problem; split-K only when the experts' tiles cannot fill the GPU.
fp8bq_variant default_grouped_variant(int64_t E, int64_t M, int64_t N, int64_t K, int fmt,
                                      int num_sms) {
    fp8bq_variant v = {};
    int64_t tiles;
    if (M <= 128) {
        v.kind = FP8BQ_KIND_SWAP_AB;
        v.block_n = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
        tiles = E * (N / 128) * ((M + v.block_n - 1) / v.block_n);
    } else {
        v.kind = FP8BQ_KIND_NORMAL;
        v.block_n = N % 256 == 0 ? 256 : 128;
        tiles = E * (N / v.block_n) * ((M + 127) / 128);
    }
    const int64_t G = K / kGroup;
    int64_t split = 1;
    if (tiles > 0 && tiles < num_sms && tiles * 8 * 4 <= static_cast<int64_t>(kCounterRegion)) {
        split = (num_sms + tiles - 1) / tiles;
        if (split > 8) split = 8;
        if (split > G) split = G;
    }
    v.split = static_cast<int>(split);
    v.grid = 0;
    v.mma_scale = (fmt == FP8BQ_SCALE_UE8M0 && K % (4 * kGroup) == 0 &&
                   (v.kind == FP8BQ_KIND_NORMAL || v.block_n >= 64))
                      ? 1
                      : 0;
    v.from_table = 0;
    return v;
}

// ------------------------------------------------------- argument checks

constexpr int64_t kMaxDim = (1LL << 31) - 4096;

fp8bq_status check_gemm_args(int64_t M, int64_t N, int64_t K, int fmt, int out_dtype) {
    if (M < 0 || N < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (fmt != FP8BQ_SCALE_FP32 && fmt != FP8BQ_SCALE_UE8M0) return FP8BQ_ERR_INVALID_ARG;
    if (out_dtype != FP8BQ_BF16 && out_dtype != FP8BQ_FP16 && out_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_INVALID_ARG;
    if (K == 0 || K % 128 != 0 || N % 64 != 0) return FP8BQ_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    return FP8BQ_OK;
}

fp8bq_status check_gemm_ptrs(const void* a_q, const void* a_s, const void* w_q, const void* w_s,
                             const void* out) {
    if (!a_q || !a_s || !w_q || !w_s || !out) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(w_q) || !aligned16(w_s) ||
        !aligned16(out))
        return FP8BQ_ERR_ALIGNMENT;
    return FP8BQ_OK;
}

fp8bq_status check_ws(const GemmPlan& plan, const void* ws, size_t ws_bytes) {
    if (plan.ws_bytes == 0) return FP8BQ_OK;
    if (!ws || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return FP8BQ_ERR_WORKSPACE;
    return FP8BQ_OK;
}

// Grouped problems: E >= 1 experts of M_max token rows (a multiple of 4, so
// every expert's scale rows start on a 16-byte boundary), weights in whole
// 128-row blocks per expert (N % 128 == 0).
fp8bq_status check_grouped_args(int64_t E, int64_t M_max, int64_t N, int64_t K, int fmt,
                                int out_dtype) {
    if (E < 1 || E > (1 << 20) || M_max < 0) return FP8BQ_ERR_INVALID_ARG;
    if (M_max > kMaxDim / E || N > kMaxDim / E) return FP8BQ_ERR_SHAPE;
    fp8bq_status st = check_gemm_args(E * M_max, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (M_max % 4 != 0 || N % kGroup != 0) return FP8BQ_ERR_SHAPE;
    return FP8BQ_OK;
}

// Rowwise (per-token x per-channel) formats: K in whole 16-byte code rows,
// N a multiple of 16 (16-byte aligned output rows for every dtype).
fp8bq_status check_rowwise_args(int64_t M, int64_t N, int64_t K, int code, int out_dtype) {
    if (M < 0 || N < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (code != FP8BQ_CODE_E4M3 && code != FP8BQ_CODE_INT8) return FP8BQ_ERR_INVALID_ARG;
    if (out_dtype != FP8BQ_BF16 && out_dtype != FP8BQ_FP16 && out_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_INVALID_ARG;
    if (K == 0 || K % 16 != 0 || N % 16 != 0) return FP8BQ_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    return FP8BQ_OK;
}

fp8bq_status check_rowwise_ptrs(const void* a_q, const float* a_s, const void* w_q,
                                const float* w_s, const void* out) {
    if (!a_q || !a_s || !w_q || !w_s || !out) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(w_q) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(a_s) & 3u) || (reinterpret_cast<uintptr_t>(w_s) & 3u))
        return FP8BQ_ERR_ALIGNMENT;
    return FP8BQ_OK;
}

// INT8 shapes without a measured table entry: at least this many tokens run
// as two e4m3 planes on the tcgen05 FP8 MMA (four cross products per K step),
// fewer on the warp-level int8 MMA, which streams the int8 weights once.  The
// warp-level kernel wins while one token tile covers M and the int8 MMA rate
// is not yet the bound; where the two are close (48-64 tokens on GB300) the
// table's measured entries decide.
constexpr int64_t kInt8PlanesMinM = 65;

// Kernel shape of a rowwise problem.  e4m3: the tile and split the block path
// uses for UE8M0 scales (its table when it has the shape; the rowwise kernel
// is the block-scaled one without factors), on the promotion-free kernel.
// int8, M >= kInt8PlanesMinM: the default variant's tiles with mma_scale = 1
// (the FP8-plane kernel); smaller M: swap-AB with the token tile covering M.
fp8bq_variant rowwise_variant(int64_t M, int64_t N, int64_t K, int code, int out_dtype,
                              const std::string& device_name, int num_sms) {
    // shapes measured for the rowwise kernels themselves (checked as the
    // planner would: a stale or hand-edited entry falls through)
    fp8bq_variant measured;
    const int tfmt = code == FP8BQ_CODE_E4M3 ? kTableRowwiseE4m3 : kTableRowwiseInt8;
    if (format_table_lookup(tfmt, M, N, K, out_dtype, device_name, &measured)) {
        GemmPlan probe;
        const int mode = code == FP8BQ_CODE_E4M3 ? 1 : (measured.mma_scale ? 3 : 2);
        const int64_t Kg = mode == 3 ? (K + kGroup - 1) / kGroup * kGroup : K;
        if (make_gemm_plan(M, N, Kg, measured, num_sms, &probe, 0, mode)) return measured;
    }
    fp8bq_variant v = code == FP8BQ_CODE_E4M3
                          ? select_variant(M, N, K, FP8BQ_SCALE_UE8M0, out_dtype, device_name,
                                           num_sms)
                          : default_variant(M, N, K, FP8BQ_SCALE_FP32, num_sms);
    v.mma_scale = 0;
    if (v.kind == FP8BQ_KIND_SWAP_AB_64) v.kind = FP8BQ_KIND_SWAP_AB;
    if (code == FP8BQ_CODE_INT8 && M >= kInt8PlanesMinM) {
        v.mma_scale = 1;
        // whole tiles: stream-K shares re-read the planes' doubled operands
        // (2048 x 7168 x 18432 on GB300: 866 us stream-K, 650 us whole tiles)
        if (v.kind == FP8BQ_KIND_NORMAL) v.split = 1;
    } else if (code == FP8BQ_CODE_INT8 && M <= 8) {
        // an 8-token tile halves the int8 MMA work, which bounds 16-token
        // tiles even at decode sizes
        v.block_n = 8;
    } else if (code == FP8BQ_CODE_INT8 && v.kind != FP8BQ_KIND_SWAP_AB) {
        v.kind = FP8BQ_KIND_SWAP_AB;
        v.block_n = 128;
        const int64_t tiles = ((N + 127) / 128) * ((M + 127) / 128);
        const bool whole_waves = tiles % num_sms == 0 || tiles >= 4 * int64_t(num_sms);
        v.split = (!whole_waves && tiles * 8 * 4 <= static_cast<int64_t>(kCounterRegion)) ? 0 : 1;
        v.grid = 0;
    }
    const int64_t G = (K + kGroup - 1) / kGroup;
    if (v.split > G) v.split = static_cast<int>(G);
    return v;
}

// Rowwise kernel mode of a code and variant (GemmPlan::rowwise).
int rowwise_mode(int code, const fp8bq_variant& v) {
    if (code == FP8BQ_CODE_E4M3) return 1;
    return v.mma_scale ? 3 : 2;
}

// INT8 as e4m3 planes: K rounded up to whole slabs, two plane bytes per column.
int64_t planes_k(int64_t K) { return (K + kGroup - 1) / kGroup * kGroup; }
size_t planes_bytes(int64_t rows, int64_t K) {
    return align256(static_cast<size_t>(rows) * 2 * static_cast<size_t>(planes_k(K)));
}

fp8bq_status run_gemm(const GemmPlan& plan, int64_t M, int64_t N, int64_t K, const void* a_q,
                      const void* a_s, const void* w_q, const float* w_s, int fmt, int out_dtype,
                      void* out, void* ws, size_t ws_data_offset, DeviceInfo* d,
                      int prefetch_w, cudaStream_t stream) {
    // the block-scaled MMA takes E8M0 factors in whole groups of four slabs
    if (plan.mx && (fmt != FP8BQ_SCALE_UE8M0 || K % (4 * kGroup) != 0))
        return FP8BQ_ERR_UNSUPPORTED;
    GemmLaunch g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.a_q = a_q;
    g.a_s = a_s;
    g.w_q = w_q;
    g.w_s = w_s;
    g.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    g.out_dtype = out_dtype;
    g.out = out;
    g.workspace = ws;
    g.ws_data_offset = ws_data_offset;
    g.status = d->status;
    g.timeout_ns = wait_timeout_ns();
    g.prefetch_w = prefetch_w;
    g.x = nullptr;
    g.x_fp16 = 0;
    return from_cuda(launch_gemm(plan, g, stream));
}

fp8bq_status run_grouped_gemm(const GemmPlan& plan, int64_t E, int64_t M_max, int64_t N,
                              int64_t K, const int32_t* counts, const void* a_q, const void* a_s,
                              const void* w_q, const float* w_s, int fmt, int out_dtype,
                              void* out, void* ws, size_t ws_data_offset, DeviceInfo* d,
                              cudaStream_t stream) {
    if (plan.mx && (fmt != FP8BQ_SCALE_UE8M0 || K % (4 * kGroup) != 0))
        return FP8BQ_ERR_UNSUPPORTED;
    GemmLaunch g;
    g.M = E * M_max;
    g.N = N;
    g.K = K;
    g.a_q = a_q;
    g.a_s = a_s;
    g.w_q = w_q;
    g.w_s = w_s;
    g.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    g.out_dtype = out_dtype;
    g.out = out;
    g.workspace = ws;
    g.ws_data_offset = ws_data_offset;
    g.status = d->status;
    g.timeout_ns = wait_timeout_ns();
    g.prefetch_w = 0;
    g.x = nullptr;
    g.x_fp16 = 0;
    g.E = E;
    g.m_max = M_max;
    g.counts = counts;
    return from_cuda(launch_gemm(plan, g, stream));
}

// The linear path's fused variant: the block-scaled GEMM quantises its own
// activation tiles from x (one launch instead of quant + GEMM).
fp8bq_status run_linear_fused(const GemmPlan& plan, int64_t M, int64_t N, int64_t K,
                              const void* x, int x_fp16, const void* w_q, const float* w_s,
                              int out_dtype, void* out, void* ws, DeviceInfo* d,
                              cudaStream_t stream) {
    GemmLaunch g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.a_q = nullptr;
    g.a_s = nullptr;
    g.w_q = w_q;
    g.w_s = w_s;
    g.ue8m0 = 1;
    g.out_dtype = out_dtype;
    g.out = out;
    g.workspace = ws;
    g.ws_data_offset = 0;
    g.status = d->status;
    g.timeout_ns = wait_timeout_ns();
    g.prefetch_w = 1;
    g.x = x;
    g.x_fp16 = x_fp16;
    return from_cuda(launch_gemm(plan, g, stream));
}

// FP8BQ_LINEAR_FUSE=1 turns the fused linear variant on.  It is off by
// default: on GB300 it measured slower than quant + GEMM at every decode
// shape (each 4-slab factor group waits for all four slabs' quantisation, so
// the weight stream loses pipeline depth).  Both give the same bits.
bool linear_fuse_enabled() {
    const char* e = std::getenv("FP8BQ_LINEAR_FUSE");
    return e && e[0] == '1';
}

// Block INT8 kernel shapes.

fp8bq_status check_int8_block_args(int64_t M, int64_t N, int64_t K, int out_dtype) {
    if (M < 0 || N < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (out_dtype != FP8BQ_BF16 && out_dtype != FP8BQ_FP16 && out_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_INVALID_ARG;
    if (K == 0 || K % kGroup != 0 || N % 16 != 0) return FP8BQ_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    return FP8BQ_OK;
}

// swap-AB on the warp-level int8 MMA: the token tile covering M (8 up to 8
// tokens), 128-token tiles above 128; split-K / stream-K as the FP8 default
fp8bq_variant int8_block_variant(int64_t M, int64_t N, int64_t K, int out_dtype, int num_sms,
                                 const std::string& device_name) {
    fp8bq_variant measured;
    if (format_table_lookup(kTableBlockInt8, M, N, K, out_dtype, device_name, &measured)) {
        GemmPlan probe;
        if (make_gemm_plan(M, N, K, measured, num_sms, &probe, 0, measured.mma_scale ? 5 : 4))
            return measured;
    }
    fp8bq_variant v = default_variant(M, N, K, FP8BQ_SCALE_FP32, num_sms);
    if (M >= kInt8PlanesMinM) {
        // two e4m3 planes on the promotion kernel, the default tile; whole
        // tiles for the normal orientation (as the rowwise INT8 planes)
        v.mma_scale = 1;
        if (v.kind == FP8BQ_KIND_NORMAL) v.split = 1;
        return v;
    }
    v.mma_scale = 0;
    v.kind = FP8BQ_KIND_SWAP_AB;
    v.block_n = M <= 8 ? 8 : M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128;
    const int64_t tiles = ((N + 127) / 128) * ((M + v.block_n - 1) / v.block_n);
    const bool whole_waves = tiles % num_sms == 0 || tiles >= 4 * static_cast<int64_t>(num_sms);
    v.split = (!whole_waves && tiles * 8 * 4 <= static_cast<int64_t>(kCounterRegion)) ? 0 : 1;
    v.grid = 0;
    return v;
}

int host_sms() {
    DeviceInfo* d = nullptr;
    return device_info(&d) == FP8BQ_OK ? d->num_sms : 152;  // GB300 without a visible GPU
}

std::string host_device_name() {
    DeviceInfo* d = nullptr;
    return device_info(&d) == FP8BQ_OK ? d->name : std::string();
}

// Kernel shape of a grouped problem: the table's grouped entry for (N, K,
// out) at the nearest rows-per-expert M_max when it has one and the planner
// (and, for the block-scaled MMA, the scale format) accepts it for these E;
// else the default rule.  The entries are measured at one expert count.
fp8bq_variant grouped_variant(int64_t E, int64_t M_max, int64_t N, int64_t K, int fmt, int out,
                              const std::string& device_name, int num_sms) {
    fp8bq_variant measured;
    const int tfmt = fmt == FP8BQ_SCALE_UE8M0 ? kTableGroupedUe8m0 : kTableGroupedFp32;
    if (format_table_lookup(tfmt, M_max, N, K, out, device_name, &measured)) {
        GemmPlan probe;
        const bool mx_ok =
            !measured.mma_scale || (fmt == FP8BQ_SCALE_UE8M0 && K % (4 * kGroup) == 0);
        if (mx_ok && make_gemm_plan(M_max, N, K, measured, num_sms, &probe, E)) return measured;
    }
    return default_grouped_variant(E, M_max, N, K, fmt, num_sms);
}

}  // namespace
}  // namespace fp8bq

using namespace fp8bq;

// =========================================================== C ABI

extern "C" {

int fp8bq_abi_version(void) { return 1; }

const char* fp8bq_status_string(fp8bq_status s) {
    switch (s) {
        case FP8BQ_OK: return "ok";
        case FP8BQ_ERR_INVALID_ARG: return "invalid argument";
        case FP8BQ_ERR_SHAPE: return "unsupported shape (K must be a positive multiple of 128, N of 64)";
        case FP8BQ_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case FP8BQ_ERR_UNSUPPORTED: return "unsupported group/block size, dtype or GPU";
        case FP8BQ_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case FP8BQ_ERR_LAUNCH: return "kernel launch failed";
        case FP8BQ_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
        case FP8BQ_ERR_CUDA: return "CUDA runtime error";
    }
    return "unknown status";
}

size_t fp8bq_act_scale_bytes(int64_t M, int64_t K, int group, fp8bq_scale_fmt fmt) {
    if (M < 0 || K <= 0 || group != kGroup || K % group) return 0;
    if (fmt != FP8BQ_SCALE_FP32 && fmt != FP8BQ_SCALE_UE8M0) return 0;
    const int64_t G = K / group;
    const int64_t cols = fmt == FP8BQ_SCALE_UE8M0 ? (G + 3) / 4 : G;
    return static_cast<size_t>(4 * cols * pad_rows4(M));
}

size_t fp8bq_weight_scale_bytes(int64_t N, int64_t K, int block_n, int block_k) {
    if (N < 0 || K <= 0 || block_n != kGroup || block_k != kGroup || K % block_k) return 0;
    return static_cast<size_t>(4 * ((N + block_n - 1) / block_n) * (K / block_k));
}

size_t fp8bq_variant_workspace_bytes(int64_t M, int64_t N, int64_t K, const fp8bq_variant* v) {
    if (!v || check_gemm_args(M, N, K, FP8BQ_SCALE_FP32, FP8BQ_BF16) != FP8BQ_OK) return 0;
    if (M == 0 || N == 0) return 0;
    GemmPlan plan;
    if (!make_gemm_plan(M, N, K, *v, host_sms(), &plan)) return 0;
    return plan.ws_bytes;
}

fp8bq_status fp8bq_variant_supported(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                     const fp8bq_variant* v) {
    if (!v) return FP8BQ_ERR_INVALID_ARG;
    fp8bq_status st = check_gemm_args(M, N, K, fmt, FP8BQ_BF16);
    if (st != FP8BQ_OK) return st;
    if (v->mma_scale && (fmt != FP8BQ_SCALE_UE8M0 || K % (4 * kGroup) != 0))
        return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    GemmPlan plan;
    return make_gemm_plan(M, N, K, *v, host_sms(), &plan) ? FP8BQ_OK : FP8BQ_ERR_UNSUPPORTED;
}

fp8bq_status fp8bq_select_variant(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                  fp8bq_dtype out_dtype, fp8bq_variant* variant) {
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    fp8bq_status st = check_gemm_args(M, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    std::string name;
    int sms = 152;  // GB300 when no GPU is visible (host-only queries)
    if (device_info(&d) == FP8BQ_OK) {
        name = d->name;
        sms = d->num_sms;
    }
    *variant = select_variant(M, N, K, fmt, out_dtype, name, sms);
    return FP8BQ_OK;
}

fp8bq_status fp8bq_reload_table(void) {
    std::lock_guard<std::mutex> lock(g_table_mutex);
    g_table.loaded = false;
    return FP8BQ_OK;
}

size_t fp8bq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                  fp8bq_dtype out_dtype) {
    fp8bq_variant v;
    if (fp8bq_select_variant(M, N, K, fmt, out_dtype, &v) != FP8BQ_OK) return 0;
    return fp8bq_variant_workspace_bytes(M, N, K, &v);
}

size_t fp8bq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                    fp8bq_dtype out_dtype) {
    if (check_gemm_args(M, N, K, fmt, out_dtype) != FP8BQ_OK) return 0;
    const size_t g = fp8bq_gemm_workspace_bytes(M, N, K, fmt, out_dtype);
    return kCounterRegion + align256(static_cast<size_t>(M * K)) +
           align256(fp8bq_act_scale_bytes(M, K, kGroup, fmt)) + (g ? g - kCounterRegion : 0);
}

fp8bq_status fp8bq_quant_act(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t K, int group,
                             fp8bq_scale_fmt fmt, void* q, void* s, cudaStream_t stream) {
    if (M < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (fmt != FP8BQ_SCALE_FP32 && fmt != FP8BQ_SCALE_UE8M0) return FP8BQ_ERR_INVALID_ARG;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (group != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (K == 0 || K % kGroup != 0 || K > kMaxDim || M > kMaxDim) return FP8BQ_ERR_SHAPE;
    if (M == 0) return FP8BQ_OK;
    if (!x || !q || !s) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return FP8BQ_ERR_ALIGNMENT;
    if ((K / kGroup + 3) / 4 > 65535) return FP8BQ_ERR_SHAPE;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    QuantActArgs a;
    a.x = x;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.M = M;
    a.Mp = pad_rows4(M);
    a.K = K;
    a.G = static_cast<int>(K / kGroup);
    a.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    a.fp16 = x_dtype == FP8BQ_FP16;
    return from_cuda(launch_quant_act(a, stream));
}

fp8bq_status fp8bq_quant_weight(const void* w, fp8bq_dtype w_dtype, int64_t N, int64_t K,
                                int block_n, int block_k, fp8bq_scale_fmt fmt, void* q, float* s,
                                cudaStream_t stream) {
    if (N < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (fmt != FP8BQ_SCALE_FP32 && fmt != FP8BQ_SCALE_UE8M0) return FP8BQ_ERR_INVALID_ARG;
    if (w_dtype != FP8BQ_BF16 && w_dtype != FP8BQ_FP16 && w_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_UNSUPPORTED;
    if (block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (K == 0 || K % kGroup != 0 || K > kMaxDim || N > kMaxDim) return FP8BQ_ERR_SHAPE;
    if ((N + kGroup - 1) / kGroup > 65535) return FP8BQ_ERR_SHAPE;
    if (N == 0) return FP8BQ_OK;
    if (!w || !q || !s) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(s)) return FP8BQ_ERR_ALIGNMENT;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    QuantWeightArgs a;
    a.w = w;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.N = N;
    a.K = K;
    a.NB = static_cast<int>((N + kGroup - 1) / kGroup);
    a.KB = static_cast<int>(K / kGroup);
    a.dtype = w_dtype;
    a.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    return from_cuda(launch_quant_weight(a, stream));
}

fp8bq_status fp8bq_gemm_variant(int64_t M, int64_t N, int64_t K, const void* a_q, const void* a_s,
                                const void* w_q, const float* w_s, fp8bq_scale_fmt fmt,
                                fp8bq_dtype out_dtype, void* out, const fp8bq_variant* variant,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_gemm_args(M, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_gemm_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    GemmPlan plan;
    if (!make_gemm_plan(M, N, K, *variant, d->num_sms, &plan)) return FP8BQ_ERR_UNSUPPORTED;
    st = check_ws(plan, workspace, workspace_bytes);
    if (st != FP8BQ_OK) return st;
    return run_gemm(plan, M, N, K, a_q, a_s, w_q, w_s, fmt, out_dtype, out, workspace, 0, d, 0,
                    stream);
}

fp8bq_status fp8bq_gemm(int64_t M, int64_t N, int64_t K, const void* a_q, const void* a_s,
                        const void* w_q, const float* w_s, int group, int block_n, int block_k,
                        fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_gemm_args(M, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_gemm_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = select_variant(M, N, K, fmt, out_dtype, d->name, d->num_sms);
    GemmPlan plan;
    if (!make_gemm_plan(M, N, K, v, d->num_sms, &plan)) return FP8BQ_ERR_UNSUPPORTED;
    st = check_ws(plan, workspace, workspace_bytes);
    if (st != FP8BQ_OK) return st;
    return run_gemm(plan, M, N, K, a_q, a_s, w_q, w_s, fmt, out_dtype, out, workspace, 0, d, 0,
                    stream);
}

// ------------------------------------------------------------ grouped GEMM

size_t fp8bq_grouped_variant_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                             const fp8bq_variant* v) {
    if (!v || check_grouped_args(E, M_max, N, K, FP8BQ_SCALE_FP32, FP8BQ_BF16) != FP8BQ_OK)
        return 0;
    if (M_max == 0 || N == 0) return 0;
    GemmPlan plan;
    if (!make_gemm_plan(M_max, N, K, *v, host_sms(), &plan, E)) return 0;
    return plan.ws_bytes;
}

fp8bq_status fp8bq_select_grouped_variant(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                          fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype,
                                          fp8bq_variant* variant) {
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    fp8bq_status st = check_grouped_args(E, M_max, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    *variant = grouped_variant(E, M_max, N, K, fmt, out_dtype, host_device_name(), host_sms());
    return FP8BQ_OK;
}

size_t fp8bq_grouped_gemm_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                          fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype) {
    fp8bq_variant v;
    if (fp8bq_select_grouped_variant(E, M_max, N, K, fmt, out_dtype, &v) != FP8BQ_OK) return 0;
    return fp8bq_grouped_variant_workspace_bytes(E, M_max, N, K, &v);
}

fp8bq_status fp8bq_grouped_gemm_variant(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                        const int32_t* counts, const void* a_q, const void* a_s,
                                        const void* w_q, const float* w_s, fp8bq_scale_fmt fmt,
                                        fp8bq_dtype out_dtype, void* out,
                                        const fp8bq_variant* variant, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_grouped_args(E, M_max, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    if (M_max == 0 || N == 0) return FP8BQ_OK;
    if (!counts) return FP8BQ_ERR_INVALID_ARG;
    st = check_gemm_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    GemmPlan plan;
    if (!make_gemm_plan(M_max, N, K, *variant, d->num_sms, &plan, E)) return FP8BQ_ERR_UNSUPPORTED;
    st = check_ws(plan, workspace, workspace_bytes);
    if (st != FP8BQ_OK) return st;
    return run_grouped_gemm(plan, E, M_max, N, K, counts, a_q, a_s, w_q, w_s, fmt, out_dtype, out,
                            workspace, 0, d, stream);
}

fp8bq_status fp8bq_grouped_gemm(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                const int32_t* counts, const void* a_q, const void* a_s,
                                const void* w_q, const float* w_s, int group, int block_n,
                                int block_k, fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_grouped_args(E, M_max, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (M_max == 0 || N == 0) return FP8BQ_OK;
    fp8bq_variant v;
    st = fp8bq_select_grouped_variant(E, M_max, N, K, fmt, out_dtype, &v);
    if (st != FP8BQ_OK) return st;
    return fp8bq_grouped_gemm_variant(E, M_max, N, K, counts, a_q, a_s, w_q, w_s, fmt, out_dtype,
                                      out, &v, workspace, workspace_bytes, stream);
}

size_t fp8bq_grouped_linear_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                            fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype) {
    if (check_grouped_args(E, M_max, N, K, fmt, out_dtype) != FP8BQ_OK) return 0;
    const int64_t rows = E * M_max;
    const size_t g = fp8bq_grouped_gemm_workspace_bytes(E, M_max, N, K, fmt, out_dtype);
    return kCounterRegion + align256(static_cast<size_t>(rows * K)) +
           align256(fp8bq_act_scale_bytes(rows, K, kGroup, fmt)) + (g ? g - kCounterRegion : 0);
}

fp8bq_status fp8bq_grouped_linear(const void* x, fp8bq_dtype x_dtype, int64_t E, int64_t M_max,
                                  int64_t N, int64_t K, const int32_t* counts, const void* w_q,
                                  const float* w_s, int group, int block_n, int block_k,
                                  fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_grouped_args(E, M_max, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (E > 65535) return FP8BQ_ERR_UNSUPPORTED;  // the quant grid's expert dimension
    if (M_max == 0 || N == 0) return FP8BQ_OK;
    if (!x || !counts) return FP8BQ_ERR_INVALID_ARG;
    st = check_gemm_ptrs(x, x, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    if ((K / kGroup + 3) / 4 > 65535) return FP8BQ_ERR_SHAPE;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8BQ_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = grouped_variant(E, M_max, N, K, fmt, out_dtype, d->name, d->num_sms);
    GemmPlan plan;
    if (!make_gemm_plan(M_max, N, K, v, d->num_sms, &plan, E)) return FP8BQ_ERR_UNSUPPORTED;
    // workspace: [counter prefix][codes][scales][split-K partials], as fp8bq_linear
    const int64_t rows = E * M_max;
    const size_t q_bytes = align256(static_cast<size_t>(rows * K));
    const size_t s_bytes = align256(fp8bq_act_scale_bytes(rows, K, kGroup, fmt));
    const size_t part_bytes = plan.ws_bytes ? plan.ws_bytes - kCounterRegion : 0;
    if (workspace_bytes < kCounterRegion + q_bytes + s_bytes + part_bytes)
        return FP8BQ_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* a_q = base + kCounterRegion;
    void* a_s = base + kCounterRegion + q_bytes;
    QuantActArgs qa;
    qa.x = x;
    qa.q = static_cast<uint8_t*>(a_q);
    qa.s = a_s;
    qa.M = rows;
    qa.Mp = pad_rows4(rows);
    qa.K = K;
    qa.G = static_cast<int>(K / kGroup);
    qa.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    qa.fp16 = x_dtype == FP8BQ_FP16;
    qa.counts = counts;
    qa.m_max = M_max;
    st = from_cuda(launch_quant_act(qa, stream));
    if (st != FP8BQ_OK) return st;
    return run_grouped_gemm(plan, E, M_max, N, K, counts, a_q, a_s, w_q, w_s, fmt, out_dtype, out,
                            base, q_bytes + s_bytes, d, stream);
}

fp8bq_status fp8bq_linear(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N, int64_t K,
                          const void* w_q, const float* w_s, int group, int block_n, int block_k,
                          fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_gemm_args(M, N, K, fmt, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    if (!x) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(x)) return FP8BQ_ERR_ALIGNMENT;
    st = check_gemm_ptrs(x, x, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8BQ_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = select_variant(M, N, K, fmt, out_dtype, d->name, d->num_sms);
    GemmPlan plan;
    if (!make_gemm_plan(M, N, K, v, d->num_sms, &plan)) return FP8BQ_ERR_UNSUPPORTED;
    // workspace: [counter prefix][codes][scales][split-K partials]; the GEMM
    // sees a workspace whose prefix is the counters and whose partials follow
    // the scales, so it is passed as a base pointer with the data shifted.
    const size_t q_bytes = align256(static_cast<size_t>(M * K));
    const size_t s_bytes = align256(fp8bq_act_scale_bytes(M, K, kGroup, fmt));
    const size_t part_bytes = plan.ws_bytes ? plan.ws_bytes - kCounterRegion : 0;
    if (workspace_bytes < kCounterRegion + q_bytes + s_bytes + part_bytes)
        return FP8BQ_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* a_q = base + kCounterRegion;
    void* a_s = base + kCounterRegion + q_bytes;

    // UE8M0 with a swap-AB tile of 16/32 tokens: one block-scaled launch that
    // quantises its own activation tiles (same codes, scales and sums as the
    // two-launch path: bit-identical output to quant + block-scaled GEMM).
    if (fmt == FP8BQ_SCALE_UE8M0 && v.kind == FP8BQ_KIND_SWAP_AB && v.block_n <= 32 &&
        linear_fuse_enabled()) {
        fp8bq_variant fv = v;
        fv.mma_scale = 1;
        GemmPlan fplan;
        if (!make_gemm_plan(M, N, K, fv, d->num_sms, &fplan)) return FP8BQ_ERR_UNSUPPORTED;
        return run_linear_fused(fplan, M, N, K, x, x_dtype == FP8BQ_FP16, w_q, w_s, out_dtype,
                                out, base, d, stream);
    }

    QuantActArgs qa;
    qa.x = x;
    qa.q = static_cast<uint8_t*>(a_q);
    qa.s = a_s;
    qa.M = M;
    qa.Mp = pad_rows4(M);
    qa.K = K;
    qa.G = static_cast<int>(K / kGroup);
    qa.ue8m0 = fmt == FP8BQ_SCALE_UE8M0;
    qa.fp16 = x_dtype == FP8BQ_FP16;
    st = from_cuda(launch_quant_act(qa, stream));
    if (st != FP8BQ_OK) return st;
    return run_gemm(plan, M, N, K, a_q, a_s, w_q, w_s, fmt, out_dtype, out, base,
                    q_bytes + s_bytes, d, 1, stream);
}

// ----------------------------------------------- per-token x per-channel

// The rowwise GEMM on a workspace region: ws_base holds [counter prefix]
// [ws_skip bytes used by the caller][split parts][planes (INT8 on FP8)].
//   mode: GemmPlan::rowwise (3 and 5 rewrite both operands as INT8 planes).
fp8bq_status run_rowwise(int64_t M, int64_t N, int64_t K, const void* a_q, const float* a_s,
                         const void* w_q, const float* w_s, int mode, int out_dtype, void* out,
                         const fp8bq_variant& v, uint8_t* ws_base, size_t ws_bytes,
                         size_t ws_skip, DeviceInfo* d, int prefetch_w, cudaStream_t stream) {
    const bool planes = mode == 3 || mode == 5;
    const int64_t Kg = planes ? planes_k(K) : K;  // the GEMM's K
    GemmPlan plan;
    if (!make_gemm_plan(M, N, Kg, v, d->num_sms, &plan, 0, mode)) return FP8BQ_ERR_UNSUPPORTED;
    if (!planes) {
        if (plan.ws_bytes && (!ws_base || ws_bytes < plan.ws_bytes + ws_skip ||
                              (reinterpret_cast<uintptr_t>(ws_base) & 255u)))
            return FP8BQ_ERR_WORKSPACE;
        return run_gemm(plan, M, N, K, a_q, a_s, w_q, w_s, FP8BQ_SCALE_FP32, out_dtype, out,
                        ws_base, ws_skip, d, prefetch_w, stream);
    }
    // INT8 as e4m3 planes: both operands are rewritten into the workspace
    // first, so the GEMM may not read weights before its predecessor ends
    const size_t parts = plan.ws_bytes ? plan.ws_bytes - kCounterRegion : 0;
    const size_t a_off = align256(kCounterRegion + ws_skip + parts);
    const size_t need = a_off + planes_bytes(M, K) + planes_bytes(N, K);
    if (!ws_base || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws_base) & 255u))
        return FP8BQ_ERR_WORKSPACE;
    uint8_t* pa = ws_base + a_off;
    uint8_t* pw = pa + planes_bytes(M, K);
    Int8PlanesArgs ia;
    ia.q = static_cast<const int8_t*>(a_q);
    ia.planes = pa;
    ia.R = M;
    ia.K = K;
    ia.Kp = planes_k(K);
    fp8bq_status st = from_cuda(launch_int8_planes(ia, stream));
    if (st != FP8BQ_OK) return st;
    ia.q = static_cast<const int8_t*>(w_q);
    ia.planes = pw;
    ia.R = N;
    st = from_cuda(launch_int8_planes(ia, stream));
    if (st != FP8BQ_OK) return st;
    return run_gemm(plan, M, N, Kg, pa, a_s, pw, w_s, FP8BQ_SCALE_FP32, out_dtype, out, ws_base,
                    ws_skip, d, 0, stream);
}

fp8bq_status fp8bq_quant_rows(const void* x, fp8bq_dtype x_dtype, int64_t R, int64_t K,
                              fp8bq_code code, void* q, float* s, cudaStream_t stream) {
    if (R < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16 && x_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_INVALID_ARG;
    if (code != FP8BQ_CODE_E4M3 && code != FP8BQ_CODE_INT8) return FP8BQ_ERR_INVALID_ARG;
    if (K == 0 || K % 16 != 0 || R > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    if (R == 0) return FP8BQ_OK;
    if (!x || !q || !s) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s) & 3u))
        return FP8BQ_ERR_ALIGNMENT;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    QuantRowsArgs a;
    a.x = x;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.R = R;
    a.K = K;
    a.dtype = x_dtype;
    a.int8 = code == FP8BQ_CODE_INT8;
    return from_cuda(launch_quant_rows(a, stream));
}

size_t fp8bq_rowwise_variant_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                             const fp8bq_variant* v) {
    if (!v || check_rowwise_args(M, N, K, code, FP8BQ_BF16) != FP8BQ_OK) return 0;
    DeviceInfo* d = nullptr;
    int sms = 152;  // GB300 when no GPU is visible (host-only queries)
    if (device_info(&d) == FP8BQ_OK) sms = d->num_sms;
    const int mode = rowwise_mode(code, *v);
    GemmPlan plan;
    if (!make_gemm_plan(M, N, mode == 3 ? planes_k(K) : K, *v, sms, &plan, 0, mode)) return 0;
    if (mode != 3) return plan.ws_bytes;
    // [counter prefix][split parts][token planes][weight planes]
    const size_t base = plan.ws_bytes ? plan.ws_bytes : kCounterRegion;
    return align256(base) + planes_bytes(M, K) + planes_bytes(N, K);
}

fp8bq_status fp8bq_select_rowwise_variant(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                          fp8bq_dtype out_dtype, fp8bq_variant* variant) {
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    fp8bq_status st = check_rowwise_args(M, N, K, code, out_dtype);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    std::string name;
    int sms = 152;  // GB300 when no GPU is visible (host-only queries)
    if (device_info(&d) == FP8BQ_OK) {
        name = d->name;
        sms = d->num_sms;
    }
    *variant = rowwise_variant(M, N, K, code, out_dtype, name, sms);
    return FP8BQ_OK;
}

size_t fp8bq_rowwise_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                     fp8bq_dtype out_dtype) {
    fp8bq_variant v;
    if (fp8bq_select_rowwise_variant(M, N, K, code, out_dtype, &v) != FP8BQ_OK) return 0;
    return fp8bq_rowwise_variant_workspace_bytes(M, N, K, code, &v);
}

fp8bq_status fp8bq_gemm_rowwise_variant(int64_t M, int64_t N, int64_t K, const void* a_q,
                                        const float* a_s, const void* w_q, const float* w_s,
                                        fp8bq_code code, fp8bq_dtype out_dtype, void* out,
                                        const fp8bq_variant* variant, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_rowwise_args(M, N, K, code, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_rowwise_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    return run_rowwise(M, N, K, a_q, a_s, w_q, w_s, rowwise_mode(code, *variant), out_dtype, out,
                       *variant, static_cast<uint8_t*>(workspace), workspace_bytes, 0, d, 0,
                       stream);
}

fp8bq_status fp8bq_gemm_rowwise(int64_t M, int64_t N, int64_t K, const void* a_q,
                                const float* a_s, const void* w_q, const float* w_s,
                                fp8bq_code code, fp8bq_dtype out_dtype, void* out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_rowwise_args(M, N, K, code, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_rowwise_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = rowwise_variant(M, N, K, code, out_dtype, d->name, d->num_sms);
    return fp8bq_gemm_rowwise_variant(M, N, K, a_q, a_s, w_q, w_s, code, out_dtype, out, &v,
                                      workspace, workspace_bytes, stream);
}

size_t fp8bq_linear_rowwise_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                            fp8bq_dtype out_dtype) {
    if (check_rowwise_args(M, N, K, code, out_dtype) != FP8BQ_OK) return 0;
    // the GEMM's own layout (parts, then INT8 planes, at 256-byte offsets)
    // follows the codes and scales, so its byte count carries over
    const size_t g = fp8bq_rowwise_workspace_bytes(M, N, K, code, out_dtype);
    return kCounterRegion + align256(static_cast<size_t>(M * K)) +
           align256(static_cast<size_t>(4 * M)) + (g ? g - kCounterRegion : 0);
}

fp8bq_status fp8bq_linear_rowwise(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N,
                                  int64_t K, const void* w_q, const float* w_s, fp8bq_code code,
                                  fp8bq_dtype out_dtype, void* out, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_rowwise_args(M, N, K, code, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    if (!x) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(x)) return FP8BQ_ERR_ALIGNMENT;
    st = check_rowwise_ptrs(x, w_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8BQ_ERR_WORKSPACE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = rowwise_variant(M, N, K, code, out_dtype, d->name, d->num_sms);
    // workspace: [counter prefix][codes][scales][split parts][planes (INT8 on FP8)]
    const size_t q_bytes = align256(static_cast<size_t>(M * K));
    const size_t s_bytes = align256(static_cast<size_t>(4 * M));
    if (workspace_bytes < kCounterRegion + q_bytes + s_bytes) return FP8BQ_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* a_q = base + kCounterRegion;
    float* a_s = reinterpret_cast<float*>(base + kCounterRegion + q_bytes);
    QuantRowsArgs qa;
    qa.x = x;
    qa.q = static_cast<uint8_t*>(a_q);
    qa.s = a_s;
    qa.R = M;
    qa.K = K;
    qa.dtype = x_dtype;
    qa.int8 = code == FP8BQ_CODE_INT8;
    // check the GEMM's share of the workspace before launching anything
    const size_t need = fp8bq_linear_rowwise_workspace_bytes(M, N, K, code, out_dtype);
    if (need == 0 || workspace_bytes < need) return FP8BQ_ERR_WORKSPACE;
    st = from_cuda(launch_quant_rows(qa, stream));
    if (st != FP8BQ_OK) return st;
    return run_rowwise(M, N, K, a_q, a_s, w_q, w_s, rowwise_mode(code, v), out_dtype, out, v,
                       base, workspace_bytes, q_bytes + s_bytes, d, 1, stream);
}

// ------------------------------------------------------------ block INT8

fp8bq_status fp8bq_quant_act_int8(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t K,
                                  int group, void* q, float* s, cudaStream_t stream) {
    if (M < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (group != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (K == 0 || K % kGroup != 0 || M > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    if ((K / kGroup + 3) / 4 > 65535) return FP8BQ_ERR_SHAPE;
    if (M == 0) return FP8BQ_OK;
    if (!x || !q || !s) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(s)) return FP8BQ_ERR_ALIGNMENT;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    QuantActArgs a;
    a.x = x;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.M = M;
    a.Mp = pad_rows4(M);
    a.K = K;
    a.G = static_cast<int>(K / kGroup);
    a.ue8m0 = 0;
    a.fp16 = x_dtype == FP8BQ_FP16;
    a.int8 = 1;
    return from_cuda(launch_quant_act(a, stream));
}

fp8bq_status fp8bq_quant_weight_int8(const void* w, fp8bq_dtype w_dtype, int64_t N, int64_t K,
                                     int block_n, int block_k, void* q, float* s,
                                     cudaStream_t stream) {
    if (N < 0 || K < 0) return FP8BQ_ERR_INVALID_ARG;
    if (block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (w_dtype != FP8BQ_BF16 && w_dtype != FP8BQ_FP16 && w_dtype != FP8BQ_FP32)
        return FP8BQ_ERR_INVALID_ARG;
    if (K == 0 || K % kGroup != 0 || N > kMaxDim || K > kMaxDim) return FP8BQ_ERR_SHAPE;
    if (N == 0) return FP8BQ_OK;
    if (!w || !q || !s) return FP8BQ_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s) & 3u))
        return FP8BQ_ERR_ALIGNMENT;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    QuantWeightArgs a;
    a.w = w;
    a.q = static_cast<uint8_t*>(q);
    a.s = s;
    a.N = N;
    a.K = K;
    a.NB = static_cast<int>((N + kGroup - 1) / kGroup);
    a.KB = static_cast<int>(K / kGroup);
    a.dtype = w_dtype;
    a.ue8m0 = 0;
    a.int8 = 1;
    return from_cuda(launch_quant_weight(a, stream));
}

fp8bq_status fp8bq_select_int8_block_variant(int64_t M, int64_t N, int64_t K,
                                             fp8bq_dtype out_dtype, fp8bq_variant* variant) {
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    fp8bq_status st = check_int8_block_args(M, N, K, out_dtype);
    if (st != FP8BQ_OK) return st;
    *variant = int8_block_variant(M, N, K, out_dtype, host_sms(), host_device_name());
    return FP8BQ_OK;
}

size_t fp8bq_int8_block_variant_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                                const fp8bq_variant* v) {
    if (!v || check_int8_block_args(M, N, K, FP8BQ_BF16) != FP8BQ_OK) return 0;
    const int mode = v->mma_scale ? 5 : 4;
    GemmPlan plan;
    if (!make_gemm_plan(M, N, K, *v, host_sms(), &plan, 0, mode)) return 0;
    if (mode == 4) return plan.ws_bytes;
    // [counter prefix][split parts][token planes][weight planes]
    const size_t base = plan.ws_bytes ? plan.ws_bytes : kCounterRegion;
    return align256(base) + planes_bytes(M, K) + planes_bytes(N, K);
}

size_t fp8bq_int8_block_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_dtype out_dtype) {
    if (check_int8_block_args(M, N, K, out_dtype) != FP8BQ_OK) return 0;
    const fp8bq_variant v = int8_block_variant(M, N, K, out_dtype, host_sms(), host_device_name());
    return fp8bq_int8_block_variant_workspace_bytes(M, N, K, &v);
}

fp8bq_status fp8bq_gemm_int8_block_variant(int64_t M, int64_t N, int64_t K, const void* a_q,
                                           const float* a_s, const void* w_q, const float* w_s,
                                           fp8bq_dtype out_dtype, void* out,
                                           const fp8bq_variant* variant, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream) {
    fp8bq_status st = check_int8_block_args(M, N, K, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (!variant) return FP8BQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_gemm_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    return run_rowwise(M, N, K, a_q, a_s, w_q, w_s, variant->mma_scale ? 5 : 4, out_dtype, out,
                       *variant, static_cast<uint8_t*>(workspace), workspace_bytes, 0, d, 0,
                       stream);
}

fp8bq_status fp8bq_gemm_int8_block(int64_t M, int64_t N, int64_t K, const void* a_q,
                                   const float* a_s, const void* w_q, const float* w_s,
                                   int group, int block_n, int block_k, fp8bq_dtype out_dtype,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream) {
    fp8bq_status st = check_int8_block_args(M, N, K, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    st = check_gemm_ptrs(a_q, a_s, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = int8_block_variant(M, N, K, out_dtype, host_sms(), host_device_name());
    return fp8bq_gemm_int8_block_variant(M, N, K, a_q, a_s, w_q, w_s, out_dtype, out, &v,
                                         workspace, workspace_bytes, stream);
}

size_t fp8bq_linear_int8_block_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                               fp8bq_dtype out_dtype) {
    if (check_int8_block_args(M, N, K, out_dtype) != FP8BQ_OK) return 0;
    const size_t g = fp8bq_int8_block_workspace_bytes(M, N, K, out_dtype);
    return kCounterRegion + align256(static_cast<size_t>(M * K)) +
           align256(fp8bq_act_scale_bytes(M, K, kGroup, FP8BQ_SCALE_FP32)) +
           (g ? g - kCounterRegion : 0);
}

fp8bq_status fp8bq_linear_int8_block(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N,
                                     int64_t K, const void* w_q, const float* w_s, int group,
                                     int block_n, int block_k, fp8bq_dtype out_dtype, void* out,
                                     void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
    fp8bq_status st = check_int8_block_args(M, N, K, out_dtype);
    if (st != FP8BQ_OK) return st;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    if (x_dtype != FP8BQ_BF16 && x_dtype != FP8BQ_FP16) return FP8BQ_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return FP8BQ_OK;
    if (!x) return FP8BQ_ERR_INVALID_ARG;
    st = check_gemm_ptrs(x, x, w_q, w_s, out);
    if (st != FP8BQ_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return FP8BQ_ERR_WORKSPACE;
    if ((K / kGroup + 3) / 4 > 65535) return FP8BQ_ERR_SHAPE;
    DeviceInfo* d = nullptr;
    st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    const fp8bq_variant v = int8_block_variant(M, N, K, out_dtype, d->num_sms, d->name);
    // workspace: [counter prefix][codes][scales][split parts][planes (two-plane kernel)]
    const size_t q_bytes = align256(static_cast<size_t>(M * K));
    const size_t s_bytes = align256(fp8bq_act_scale_bytes(M, K, kGroup, FP8BQ_SCALE_FP32));
    const size_t need = fp8bq_linear_int8_block_workspace_bytes(M, N, K, out_dtype);
    if (need == 0 || workspace_bytes < need) return FP8BQ_ERR_WORKSPACE;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* a_q = base + kCounterRegion;
    float* a_s = reinterpret_cast<float*>(base + kCounterRegion + q_bytes);
    QuantActArgs qa;
    qa.x = x;
    qa.q = static_cast<uint8_t*>(a_q);
    qa.s = a_s;
    qa.M = M;
    qa.Mp = pad_rows4(M);
    qa.K = K;
    qa.G = static_cast<int>(K / kGroup);
    qa.ue8m0 = 0;
    qa.fp16 = x_dtype == FP8BQ_FP16;
    qa.int8 = 1;
    st = from_cuda(launch_quant_act(qa, stream));
    if (st != FP8BQ_OK) return st;
    return run_rowwise(M, N, K, a_q, a_s, w_q, w_s, v.mma_scale ? 5 : 4, out_dtype, out, v, base,
                       workspace_bytes, q_bytes + s_bytes, d, 1, stream);
}

fp8bq_status fp8bq_device_status(int* code, cudaStream_t stream) {
    if (!code) return FP8BQ_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyAsync(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaMemcpyAsync(d->status, &zero, sizeof(int), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return FP8BQ_ERR_CUDA;
    }
    *code = v;
    return FP8BQ_OK;
}

fp8bq_status fp8bq_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
    if (timeout_ns == 0 || timeout_ns > 10ull * 1000 * 1000 * 1000) return FP8BQ_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    fp8bq_status st = device_info(&d);
    if (st != FP8BQ_OK) return st;
    return from_cuda(launch_wait_selftest(d->status, timeout_ns, stream));
}

}  // extern "C"

namespace fp8bq {

void log_error(const char* what) {
    static const bool on = [] {
        const char* e = std::getenv("FP8BQ_LOG");
        return e && std::atoi(e) == 1;
    }();
    if (on) std::fprintf(stderr, "fp8bq: %s\n", what);
}

EncodeTiledFn get_encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<EncodeTiledFn>(nullptr);
        }
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

}  // namespace fp8bq
