// C ABI of librowops.so: argument validation, kernel selection and launch.
// The operations themselves are documented in include/rowops.h.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "rowops.h"
#include "rowops_launch.h"

extern char** environ;  // POSIX

namespace rowops {
namespace {

int elem_bytes(rowops_dtype_t dt) { return dt == ROWOPS_F32 ? 4 : 2; }

bool valid_dtype(rowops_dtype_t dt) { return dt == ROWOPS_F32 || dt == ROWOPS_BF16; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Benchmarking knobs, read from the environment at the first call and again
// on rowops_reload_tuning() (see include/rowops.h).
enum class Family { Auto, Tma, Reg, Looped, Flat };
struct Tuning {
    int tpr = 0;
    int vpt = 0;
    Family family = Family::Auto;
    int ctas_per_sm = 0;
    int ring = 0;
    int rows = 0;  // row groups per CTA of the LayerNorm+GELU row pipeline (0: automatic)
    int online = 0;  // split-row softmax form: 0 automatic, 1 two-launch, 2 single-read, 3 row groups
    int lookahead = 0;  // single-read form's lookahead in steps (0: automatic)
    int l2 = 0;         // single-read form staged in L2
    int prefetch = 0;   // its L2 prefetch distance in rows (0: automatic)
    long long wait_ns = 0;    // device-side wait limit (0: 2 s)
    long long stall_row = -1; // test hook (see include/rowops.h)
    int sched = 0;            // full-row pipelines: 0 automatic, 1 static, 2 dynamic (cluster launch control)
    int unit_rows = 0;        // dynamic schedule: rows per group in a work unit (0: automatic)
    int bwd = 0;              // LayerNorm+GELU backward partials: 0 automatic, 1 registers, 2 tensor memory
};

// The whole value as a decimal integer, else `dflt` (unset, empty or not a number).
long long parse_int(const char* v, long long dflt) {
    if (!v || !*v) return dflt;
    char* end = nullptr;
    const long long r = std::strtoll(v, &end, 10);
    return (end && *end == '\0') ? r : dflt;
}

// One pass over the environment, looking only at ROWOPS_* entries (each call
// scans it once instead of once per knob).
Tuning read_tuning() {
    Tuning t;
    bool force_looped = false;
    const char* kernel = nullptr;
    for (char** e = environ; e && *e; ++e) {
        const char* kv = *e;
        if (std::strncmp(kv, "ROWOPS_", 7) != 0) continue;
        const char* name = kv + 7;
        const char* eq = std::strchr(name, '=');
        if (!eq) continue;
        const size_t n = size_t(eq - name);
        const char* v = eq + 1;
        auto is = [&](const char* key) { return std::strlen(key) == n && std::strncmp(name, key, n) == 0; };
        if (is("FORCE_TPR")) t.tpr = int(parse_int(v, 0));
        else if (is("FORCE_VPT")) t.vpt = int(parse_int(v, 0));
        else if (is("FORCE_LOOPED")) force_looped = parse_int(v, 0) != 0;
        else if (is("KERNEL")) kernel = v;
        else if (is("CTAS_PER_SM")) t.ctas_per_sm = int(parse_int(v, 0));
        else if (is("RING_BUFFERS")) t.ring = int(parse_int(v, 0));
        else if (is("ROWS_PER_CTA")) t.rows = int(parse_int(v, 0));
        else if (is("PERSIST_LOOKAHEAD")) t.lookahead = int(parse_int(v, 0));
        else if (is("PERSIST_L2")) t.l2 = int(parse_int(v, 0));
        else if (is("PERSIST_PREFETCH")) t.prefetch = int(parse_int(v, 0));
        else if (is("WAIT_LIMIT_NS")) t.wait_ns = std::strtoll(v, nullptr, 10);
        else if (is("TEST_STALL_ROW")) t.stall_row = std::strtoll(v, nullptr, 10);
        else if (is("UNIT_ROWS")) t.unit_rows = int(parse_int(v, 0));
        else if (is("SCHED")) t.sched = !std::strcmp(v, "static") ? 1 : (!std::strcmp(v, "dynamic") ? 2 : 0);
        else if (is("BWD_PARTIALS")) t.bwd = !std::strcmp(v, "registers") ? 1 : (!std::strcmp(v, "tmem") ? 2 : 0);
        else if (is("ONLINE"))
            t.online = !std::strcmp(v, "two_pass") ? 1
                     : !std::strcmp(v, "single_read") ? 2
                     : !std::strcmp(v, "row_groups") ? 3 : 0;
    }
    // ROWOPS_KERNEL, when set to a family, overrides ROWOPS_FORCE_LOOPED
    if (force_looped) t.family = Family::Looped;
    if (kernel) {
        if (!std::strcmp(kernel, "tma")) t.family = Family::Tma;
        else if (!std::strcmp(kernel, "reg")) t.family = Family::Reg;
        else if (!std::strcmp(kernel, "looped")) t.family = Family::Looped;
        else if (!std::strcmp(kernel, "flat")) t.family = Family::Flat;
    }
    return t;
}

// The process's knobs: read once, then reused (a scan of the environment per
// call cost a measurable share of a small launch's host time).
std::mutex g_tuning_mu;
bool g_tuning_loaded = false;
Tuning g_tuning;

Tuning tuning() {
    std::lock_guard<std::mutex> lk(g_tuning_mu);
    if (!g_tuning_loaded) {
        g_tuning = read_tuning();
        g_tuning_loaded = true;
    }
    return g_tuning;
}

// Checks shared by every entry point. M == 0 passes (callers then return).
rowops_status_t check_rows(const void* x, const void* y, int64_t M, int64_t N, int64_t ld,
                           rowops_dtype_t dt) {
    if (!valid_dtype(dt) || M < 0 || N < 1 || ld < N) return ROWOPS_ERR_INVALID_VALUE;
    if (N >= (int64_t(1) << 31)) return ROWOPS_ERR_UNSUPPORTED;
    if (M == 0) return ROWOPS_OK;
    if (!x || !y) return ROWOPS_ERR_INVALID_VALUE;
    const int es = elem_bytes(dt);
    if (!aligned(x, es) || !aligned(y, es)) return ROWOPS_ERR_INVALID_VALUE;
    // elements spanned, (M - 1) * ld + N, must fit in int64 bytes
    const int64_t lim = INT64_MAX / es - N;
    if (M - 1 > lim / ld) return ROWOPS_ERR_UNSUPPORTED;
    if (x != y) {
        const uintptr_t span = uintptr_t(((M - 1) * ld + N) * es);
        const uintptr_t a = reinterpret_cast<uintptr_t>(x), b = reinterpret_cast<uintptr_t>(y);
        if (a < b + span && b < a + span) return ROWOPS_ERR_INVALID_VALUE;  // partial overlap
    }
    return ROWOPS_OK;
}

// ---- per-device attributes and per-kernel caches ---------------------------
// Device error word: the row-pipeline kernels store ROWOPS_ERR_TIMEOUT here
// when a bounded wait gives up; rowops_device_status reads and clears it.
__device__ unsigned g_device_error;

struct DeviceInfo {
    unsigned long long ctx = 0;  // context the cached values belong to
    int num_sms = 0;
    int max_smem_optin = 0;
    unsigned* err = nullptr;  // device address of g_device_error on this device
    int cooperative = 0;
};

std::mutex g_mu;
std::vector<std::pair<int, DeviceInfo>> g_devices;

struct OccEntry {
    const void* func;
    unsigned long long ctx;
    int block;
    size_t smem;
    int blocks_per_sm;
};
std::vector<OccEntry> g_occ;

struct SmemEntry {
    const void* func;
    unsigned long long ctx;
    size_t smem;
};
std::vector<SmemEntry> g_smem;

cudaError_t device_info(int dev, DeviceInfo* out) {
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& d : g_devices)
        if (d.first == dev && d.second.ctx == ctx && ctx != 0) {
            *out = d.second;
            return cudaSuccess;
        }
    DeviceInfo di;
    cudaError_t e = cudaDeviceGetAttribute(&di.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&di.cooperative, cudaDevAttrCooperativeLaunch, dev);
    // (the symbol lookup also makes the device's primary context current if
    // no context was yet, so the id is taken after it)
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&di.err), g_device_error);
    if (e != cudaSuccess) return e;
    di.ctx = current_context_id();
    // one entry per device: a reset context's entry is replaced
    bool replaced = false;
    for (auto& d : g_devices)
        if (d.first == dev) {
            d.second = di;
            replaced = true;
        }
    if (!replaced) g_devices.emplace_back(dev, di);
    *out = di;
    return cudaSuccess;
}

rowops_status_t make_cfg(cudaStream_t stream, const Tuning& tn, LaunchCfg* cfg) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ROWOPS_ERR_CUDA;
    DeviceInfo di;
    if (device_info(dev, &di) != cudaSuccess) return ROWOPS_ERR_CUDA;
    cfg->stream = stream;
    cfg->device = dev;
    cfg->ctx = di.ctx;
    cfg->num_sms = di.num_sms;
    cfg->max_smem_optin = di.max_smem_optin;
    cfg->ctas_per_sm = tn.ctas_per_sm;
    cfg->dev_error = di.err;
    cfg->cooperative = di.cooperative != 0;
    cfg->persist_lookahead = tn.lookahead;
    cfg->grouped_block = tn.tpr;
    cfg->persist_l2 = tn.l2 != 0;
    cfg->persist_prefetch = tn.prefetch;
    cfg->wait_ns = tn.wait_ns > 0 ? (unsigned long long)tn.wait_ns : 2000000000ull;
    cfg->stall_row = tn.stall_row;
    // RMSNorm row pipeline on full rows (the other pipelines have a static schedule only)
    cfg->unit_rows = tn.sched == 2 ? (tn.unit_rows > 0 ? tn.unit_rows : 1) : 0;
    return ROWOPS_OK;
}

rowops_status_t finish(cudaError_t e) {
    if (e != cudaSuccess) {
        cudaGetLastError();  // the failure is reported through the status; clear it
        return ROWOPS_ERR_CUDA;
    }
    return ROWOPS_OK;
}

// Register-resident kernel choice: the smallest row group (threads per row)
// that holds floor(N / vec) 16-byte vectors with at most kMaxVpt per thread.
// The unaligned head and tail (< 2 vec elements) go one per thread, and
// every group has at least 16 threads, which covers them.
bool choose_reg(int64_t N, int es, const Tuning& tn, int* tpr_index, int* vpt) {
    const int64_t vec = 16 / es;
    const int64_t nvec = N / vec;
    if (tn.tpr) {
        int idx = -1;
        for (int i = 0; i < kNumTpr; ++i)
            if (kTprChoices[i] == tn.tpr) idx = i;
        if (idx < 0) return false;
        const int64_t need = (nvec + tn.tpr - 1) / tn.tpr;
        const int v = tn.vpt ? tn.vpt : int(need < 1 ? 1 : need);
        if (v < 1 || v > kMaxVpt || int64_t(v) * tn.tpr < nvec) return false;
        *tpr_index = idx;
        *vpt = v;
        return true;
    }
    for (int i = 0; i < kNumTpr; ++i) {
        const int64_t tpr = kTprChoices[i];
        if (tpr * kMaxVpt >= nvec) {
            const int64_t need = (nvec + tpr - 1) / tpr;
            *tpr_index = i;
            *vpt = int(need < 1 ? 1 : need);
            return true;
        }
    }
    return false;
}

bool same_phase(const void* x, const void* y) {
    return ((reinterpret_cast<uintptr_t>(x) - reinterpret_cast<uintptr_t>(y)) & 15u) == 0;
}

// batches above 32 MiB: more than L2 keeps for a few rows per SM
bool big_batch(int64_t M, int64_t N, int es) { return M * N * es > (int64_t(32) << 20); }

// The row pipeline (bulk copies through a shared-memory ring) pays its ring's
// fill latency once per CTA and a wait, its group reductions and a refill on
// every row. On a batch of at most 32 MiB (L2-resident, a few rows per SM) the
// register-resident kernels are faster (GB300, CUDA graphs: LayerNorm+GELU
// fp32 4096 x 768 6.2 us against 9.0, softmax fp32 1024 x 768 2.6 against
// 2.9), and so they are on larger batches of rows shorter than `min_row_bytes`
// (each operation's crossover, measured back to back on GB300: e.g. softmax
// fp32 262144 x 256 89 us against 248, LayerNorm+GELU bf16 131072 x 1024 120
// against 197, row sum bf16 65536 x 2048 41 against 60). Applies when the
// family is left automatic.
bool pipeline_pays(const Tuning& tn, int64_t M, int64_t N, int es, int64_t min_row_bytes) {
    if (tn.family == Family::Tma) return true;
    return tn.family == Family::Auto && big_batch(M, N, es) && N * es >= min_row_bytes;
}

// Rows from which each operation's row pipeline beats its register kernel on
// large batches (GB300): LayerNorm+GELU and RMSNorm 4 KB (bf16 65536 x 2048
// RMSNorm 84 against 105 us; 2 KB rows 91 against 95 the other way); softmax
// 8 KB in bf16 (65536 x 4096: 178 against 188 us) and 16 KB in fp32 (8 KB
// rows: 162 against 174 the other way); row sum / max 16 KB (8 KB rows: 78
// against 83 us the other way; 16 KB within 1%).
constexpr int64_t kPipeRowsNorm = 4096;
constexpr int64_t kPipeRowsReduce = 16384;
inline int64_t pipe_rows_softmax(int es) { return es == 4 ? 16384 : 8192; }

// all rows of x (and, being in phase, of y) start on 16-byte boundaries
bool rows_aligned(const void* x, const void* y, int64_t ld, int es) {
    return aligned(x, 16) && aligned(y, 16) && ((ld * es) % 16) == 0;
}

constexpr int64_t kMinChunk = 256;

// Row-pipeline kernel choice. x and y rows must share their offset modulo 16
// bytes and a row must hold at least 64 whole vectors. Rows that start on
// 16-byte boundaries with a length that fills TPR * VPT vectors exactly get the
// FULL form (no predicates), trying vectors per thread in `order` (measured on
// GB300, 8 per thread is fastest for both operations on the 4096 / 8192-column
// bf16 rows); all other rows get the general form (bulk-copied body, unaligned
// head and tail loaded directly) with the same preference among the tiles that
// leave at most 1/8 of their vector slots idle.
struct TmaChoice {
    int block_index, vpt_index;
    bool full;
};

int tma_vpt_index(int vpt) {
    for (int j = 0; j < kNumTmaVpts; ++j)
        if (kTmaVpts[j] == vpt) return j;
    return -1;
}

int tma_block_index(int64_t block) {
    for (int i = 0; i < kNumTmaBlocks; ++i)
        if (kTmaBlocks[i] == block) return i;
    return -1;
}

bool choose_tma(const void* x, const void* y, int64_t N, int64_t ld, int es, const Tuning& tn,
                std::initializer_list<int> order, TmaChoice* c) {
    const int64_t vec = 16 / es;
    if (!same_phase(x, y)) return false;
    const bool aligned = rows_aligned(x, y, ld, es) && N % vec == 0;
    const int64_t nvec = N / vec;  // the most whole vectors any row's body holds
    if (nvec < 64) return false;
    if (tn.tpr) {
        const int bi = tma_block_index(tn.tpr);
        if (bi < 0) return false;
        int vpt = tn.vpt ? tn.vpt : int((nvec + tn.tpr - 1) / tn.tpr);
        if (vpt == 5 || vpt == 6 || vpt == 7) vpt = 8;
        const int vi = tma_vpt_index(vpt);
        if (vi < 0 || int64_t(vpt) * tn.tpr < nvec) return false;
        *c = TmaChoice{bi, vi, aligned && int64_t(vpt) * tn.tpr == nvec};
        return true;
    }
    if (aligned)
        for (int vpt : order) {
            if (nvec % vpt) continue;
            const int bi = tma_block_index(nvec / vpt);
            if (bi >= 0) {
                *c = TmaChoice{bi, tma_vpt_index(vpt), true};
                return true;
            }
        }
    // general rows: the same order of vectors per thread, taking the smallest
    // block that covers the row with at most 1/8 of its vector slots idle; else
    // the combination with the fewest slots
    int best_i = -1, best_j = -1;
    int64_t best_slots = 0;
    for (int vpt : order) {
        for (int i = 0; i < kNumTmaBlocks; ++i) {
            const int64_t slots = int64_t(kTmaBlocks[i]) * vpt;
            if (slots < nvec) continue;
            if ((slots - nvec) * 8 <= slots) {
                *c = TmaChoice{i, tma_vpt_index(vpt), false};
                return true;
            }
            if (best_i < 0 || slots < best_slots) {
                best_i = i;
                best_j = tma_vpt_index(vpt);
                best_slots = slots;
            }
            break;  // larger blocks only leave more slots idle
        }
    }
    if (best_i < 0) return false;
    *c = TmaChoice{best_i, best_j, false};
    return true;
}

// Ring depth: two rows in flight per CTA by default (deeper rings measured no
// faster on GB300: the several CTAs per SM already keep enough bytes in
// flight), fewer if shared memory would not hold them next to `fixed` bytes.
// `min_slot`: a floor on the slot size (the whole tile, for kernels that keep
// the vectors past a row's body zero in every slot).
int ring_buffers(int64_t N, int es, size_t fixed, const Tuning& tn, const LaunchCfg& cfg, size_t min_slot = 0) {
    int nbuf = tn.ring > 0 ? tn.ring : 2;
    if (nbuf < 2) nbuf = 2;
    if (nbuf > 16) nbuf = 16;
    const size_t limit = size_t(cfg.max_smem_optin) - 1024;  // room for static reduction buffers
    const size_t slot = std::max(tma_row_bytes(N, es), min_slot);
    auto ring = [&](int nb) { return size_t(kTmaRingHeader) + size_t(nb) * slot; };
    while (nbuf > 2 && ring(nbuf) + fixed > limit) --nbuf;
    return ring(nbuf) + fixed <= limit ? nbuf : 0;
}

// Row groups per CTA for the LayerNorm+GELU row pipeline: the groups of a CTA
// share one staging of w, b, so packing several rows into a CTA raises the warps
// an SM can hold when that staging, not registers, limits occupancy. Picks the
// count (1, 2, 4, 5 or 8, where that instantiation exists) that gives the most
// resident warps per SM by the occupancy calculator (shared memory, registers
// and threads of the actual kernel); ties go to fewer groups.
// `ctas(rows)`: CTAs per SM of the instantiation with that many row groups (0
// if there is none or it does not fit).
template <class CtasOf>
int choose_group_rows(int tpr, int nbuf, const Tuning& tn, CtasOf ctas) {
    auto warps = [&](int rows) { return rows * nbuf > kTmaMaxSlots ? 0 : ctas(rows) * tpr * rows / 32; };
    if (tn.rows >= 1) return warps(tn.rows) > 0 ? tn.rows : 1;
    int best = 1, best_warps = warps(1);
    for (int r : {2, 4, 5, 8, 10}) {
        const int w = warps(r);
        if (w > best_warps) {
            best = r;
            best_warps = w;
        }
    }
    return best;
}

using TmaLnGeluLookup = TmaLnGeluKernel (*)(int tpr, int vpt, int rows, bool full);

int choose_ln_rows(TmaLnGeluLookup lookup, int tpr, int vpt, bool full, int64_t N, int nbuf, const Tuning& tn,
                   const LaunchCfg& cfg) {
    return choose_group_rows(tpr, nbuf, tn, [&](int rows) {
        const TmaLnGeluKernel k = lookup(tpr, vpt, rows, full);
        return k.launch ? k.ctas_per_sm(N, nbuf, cfg) : 0;
    });
}

using TmaRmsLookup = TmaRmsKernel (*)(int tpr, int vpt, int rows, bool full);

// RMSNorm (r == NULL) or fused residual + RMSNorm, arguments already checked.
rowops_status_t rms_dispatch(const void* x, const void* r, void* y, void* ro, const void* w, float eps, int64_t M,
                             int64_t N, int64_t ld, rowops_dtype_t dtype, cudaStream_t stream) {
    const bool res = r != nullptr;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    rowops_status_t st = make_cfg(stream, tn, &cfg);
    if (st != ROWOPS_OK) return st;
    // Full rows take the dynamic schedule by default: at bf16 65536 x 8192 it is
    // 10% faster than the static one for both forms (311 vs 347 us, 614 vs 677
    // us on GB300). (Softmax and LayerNorm+GELU ran 5-10% slower with it.)
    if (tn.sched == 0) cfg.unit_rows = tn.unit_rows > 0 ? tn.unit_rows : 1;
    const int es = elem_bytes(dtype);
    // every row pointer at the same offset modulo 16 bytes
    const bool phase = same_phase(x, y) && (!res || (same_phase(x, r) && same_phase(x, ro)));
    TmaChoice tc;
    if (pipeline_pays(tn, M, N, es, kPipeRowsNorm) && phase &&
        choose_tma(x, y, N, ld, es, tn, {8, 4, 2, 1}, &tc)) {
        const int tpr = kTmaBlocks[tc.block_index], vpt = kTmaVpts[tc.vpt_index];
        const int S = res ? 2 : 1;
        const size_t stage = rms_tma_stage_smem(tpr, vpt, es, tc.full);
        auto fits = [&](int nb) {
            return size_t(kTmaRingHeader) + size_t(nb) * S * tma_row_bytes(N, es) + stage + 1024 <=
                   size_t(cfg.max_smem_optin);
        };
        int nbuf = tn.ring > 0 ? (tn.ring < 2 ? 2 : (tn.ring > kTmaMaxSlots ? kTmaMaxSlots : tn.ring)) : 2;
        while (nbuf > 2 && !fits(nbuf)) --nbuf;
        if (fits(nbuf)) {
            const TmaRmsLookup lookup = dtype == ROWOPS_F32 ? (res ? rms_tma_f32_residual : rms_tma_f32_plain)
                                                            : (res ? rms_tma_bf16_residual : rms_tma_bf16_plain);
            const int rows = choose_group_rows(tpr, nbuf, tn, [&](int rr) {
                const TmaRmsKernel k = lookup(tpr, vpt, rr, tc.full);
                return k.launch ? k.ctas_per_sm(N, nbuf, cfg) : 0;
            });
            const TmaRmsKernel k = lookup(tpr, vpt, rows, tc.full);
            if (k.launch) return finish(k.launch(x, r, y, ro, w, eps, M, N, ld, nbuf, cfg));
        }
    }
    int tpr_index = 0, vpt = 0;
    RmsLaunch fn = nullptr;
    const bool smem_ok = rms_reg_smem(N, es) + 256 <= size_t(cfg.max_smem_optin);
    if (tn.family != Family::Looped && smem_ok && phase && choose_reg(N, es, tn, &tpr_index, &vpt))
        fn = dtype == ROWOPS_F32 ? rms_reg_f32(tpr_index, vpt, res) : rms_reg_bf16(tpr_index, vpt, res);
    if (!fn) fn = dtype == ROWOPS_F32 ? rms_looped_f32(res) : rms_looped_bf16(res);
    return finish(fn(x, r, y, ro, w, eps, M, N, ld, cfg));
}

// the row ranges of a and b share no byte
bool rows_disjoint(const void* a, const void* b, int64_t M, int64_t N, int64_t ld, int es) {
    const uintptr_t span = uintptr_t(((M - 1) * ld + N) * es);
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return !(pa < pb + span && pb < pa + span);
}

}  // namespace

int ctas_per_sm(const void* func, int block, size_t smem, const LaunchCfg& cfg) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& o : g_occ)
        if (o.func == func && o.ctx == cfg.ctx && o.block == block && o.smem == smem) return o.blocks_per_sm;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, func, block, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    g_occ.push_back(OccEntry{func, cfg.ctx, block, smem, n});
    return n;
}

namespace {
using CtxGetCurrentFn = int (*)(void**);                  // CUresult cuCtxGetCurrent(CUcontext*)
using CtxGetIdFn = int (*)(void*, unsigned long long*);   // CUresult cuCtxGetId(CUcontext, unsigned long long*)
std::once_flag g_ctx_fn_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
}  // namespace

unsigned long long current_context_id() {
    std::call_once(g_ctx_fn_once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    });
    if (!g_ctx_get_current || !g_ctx_get_id) return 0;
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) != 0 || ctx == nullptr || g_ctx_get_id(ctx, &id) != 0) return 0;
    return id;
}

int grid_for(const void* func, int block, size_t smem, int64_t items, const LaunchCfg& cfg) {
    int64_t cap;
    if (cfg.ctas_per_sm < 0) {
        cap = items;
    } else {
        int per_sm = cfg.ctas_per_sm;
        if (per_sm == 0) per_sm = ctas_per_sm(func, block, smem, cfg);
        if (per_sm < 1) per_sm = 1;
        cap = int64_t(per_sm) * cfg.num_sms;
    }
    int64_t g = items < cap ? items : cap;
    if (g < 1) g = 1;
    if (g > 0x7fffffff) g = 0x7fffffff;
    return int(g);
}

cudaError_t allow_smem(const void* func, size_t smem, const LaunchCfg& cfg, bool max_carveout) {
    if (smem == 0 || (smem <= 32 * 1024 && !max_carveout)) return cudaSuccess;
    std::lock_guard<std::mutex> lk(g_mu);
    for (auto& s : g_smem)
        if (s.func == func && s.ctx == cfg.ctx && s.smem >= smem) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    if (max_carveout)
        e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
    // the default limit covers static + dynamic shared memory together; opt in
    // well before the dynamic part alone reaches it
    if (e == cudaSuccess && smem > 32 * 1024)
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) g_smem.push_back(SmemEntry{func, cfg.ctx, smem});
    return e;
}

}  // namespace rowops

using namespace rowops;

extern "C" {

void rowops_reload_tuning(void) {
    const Tuning t = read_tuning();
    std::lock_guard<std::mutex> lk(g_tuning_mu);
    g_tuning = t;
    g_tuning_loaded = true;
}

const char* rowops_status_string(rowops_status_t status) {
    switch (status) {
        case ROWOPS_OK: return "ROWOPS_OK";
        case ROWOPS_ERR_INVALID_VALUE: return "ROWOPS_ERR_INVALID_VALUE";
        case ROWOPS_ERR_UNSUPPORTED: return "ROWOPS_ERR_UNSUPPORTED";
        case ROWOPS_ERR_WORKSPACE: return "ROWOPS_ERR_WORKSPACE";
        case ROWOPS_ERR_CUDA: return "ROWOPS_ERR_CUDA";
        case ROWOPS_ERR_TIMEOUT: return "ROWOPS_ERR_TIMEOUT";
    }
    return "ROWOPS_ERR_UNKNOWN";
}

rowops_status_t rowops_softmax(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                               rowops_dtype_t dtype, cudaStream_t stream) {
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st != ROWOPS_OK || M == 0) return st;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    const int es = elem_bytes(dtype);
    TmaChoice tc;
    if (pipeline_pays(tn, M, N, es, pipe_rows_softmax(es)) &&
        choose_tma(x, y, N, ld, es, tn, {8, 4, 2, 3, 1}, &tc)) {
        const int nbuf = ring_buffers(N, es, 0, tn, cfg);
        TmaSoftmaxLaunch tf = dtype == ROWOPS_F32 ? softmax_tma_f32(tc.block_index, tc.vpt_index, tc.full)
                                                  : softmax_tma_bf16(tc.block_index, tc.vpt_index, tc.full);
        if (nbuf > 0 && tf) return finish(tf(x, y, M, N, ld, nbuf, cfg));
    }
    int tpr_index = 0, vpt = 0;
    SoftmaxLaunch fn = nullptr;
    if (tn.family != Family::Looped && same_phase(x, y) && choose_reg(N, es, tn, &tpr_index, &vpt))
        fn = dtype == ROWOPS_F32 ? softmax_reg_f32(tpr_index, vpt) : softmax_reg_bf16(tpr_index, vpt);
    if (!fn) fn = dtype == ROWOPS_F32 ? softmax_looped_f32() : softmax_looped_bf16();
    return finish(fn(x, y, M, N, ld, cfg));
}

rowops_status_t rowops_softmax_causal(const void* x, void* y, int64_t M, int64_t N, int64_t ld, int64_t period,
                                      int64_t offset, rowops_dtype_t dtype, cudaStream_t stream) {
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    const int64_t lim = int64_t(1) << 62;  // keeps (r mod period) + offset + 1 in range
    if (period < 1 || offset > lim || offset < -lim) return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    const int es = elem_bytes(dtype);
    TmaChoice tc;
    // 4 vectors per thread first: on the causal bf16 32768 x 4096 input 128 x 4 ran
    // 88 us against 104 us for 64 x 8 (the best tile of the plain softmax)
    if ((tn.family == Family::Auto || tn.family == Family::Tma) &&
        choose_tma(x, y, N, ld, es, tn, {4, 8, 2, 3, 1}, &tc) && tc.full) {
        const int nbuf = ring_buffers(N, es, 0, tn, cfg);
        TmaSoftmaxCausalLaunch tf = dtype == ROWOPS_F32 ? softmax_tma_causal_f32(tc.block_index, tc.vpt_index)
                                                        : softmax_tma_causal_bf16(tc.block_index, tc.vpt_index);
        if (nbuf > 0 && tf) return finish(tf(x, y, M, N, ld, nbuf, period, offset, cfg));
    }
    const SoftmaxCausalLaunch fn = dtype == ROWOPS_F32 ? softmax_causal_looped_f32() : softmax_causal_looped_bf16();
    return finish(fn(x, y, M, N, ld, period, offset, cfg));
}

namespace {
// Row sum (op 0) / row max (op 1): arguments checked by the callers.
rowops_status_t reduce_dispatch(const void* x, float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                                int op, cudaStream_t stream) {
    const Tuning tn = tuning();
    LaunchCfg cfg;
    rowops_status_t st = make_cfg(stream, tn, &cfg);
    if (st != ROWOPS_OK) return st;
    const int es = elem_bytes(dtype);
    TmaChoice tc;
    if (pipeline_pays(tn, M, N, es, kPipeRowsReduce) &&
        choose_tma(x, x, N, ld, es, tn, {8, 4, 2, 3, 1}, &tc)) {
        const int nbuf = ring_buffers(N, es, 0, tn, cfg);
        TmaReduceLaunch tf = dtype == ROWOPS_F32 ? reduce_tma_f32(tc.block_index, tc.vpt_index, tc.full, op)
                                                 : reduce_tma_bf16(tc.block_index, tc.vpt_index, tc.full, op);
        if (nbuf > 0 && tf) return finish(tf(x, out, M, N, ld, nbuf, cfg));
    }
    int tpr_index = 0, vpt = 0;
    ReduceLaunch fn = nullptr;
    if (tn.family != Family::Looped && choose_reg(N, es, tn, &tpr_index, &vpt))
        fn = dtype == ROWOPS_F32 ? reduce_reg_f32(tpr_index, vpt, op) : reduce_reg_bf16(tpr_index, vpt, op);
    if (!fn) fn = dtype == ROWOPS_F32 ? reduce_looped_f32(op) : reduce_looped_bf16(op);
    return finish(fn(x, out, M, N, ld, cfg));
}

rowops_status_t check_reduce(const void* x, const float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype) {
    rowops_status_t st = check_rows(x, x, M, N, ld, dtype);
    if (st != ROWOPS_OK || M == 0) return st;
    if (!out || !aligned(out, 4)) return ROWOPS_ERR_INVALID_VALUE;
    // out (M floats) must not overlap the rows of x
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), oa = reinterpret_cast<uintptr_t>(out);
    const uintptr_t xspan = uintptr_t(((M - 1) * ld + N) * elem_bytes(dtype)), ospan = uintptr_t(M) * 4;
    if (xa < oa + ospan && oa < xa + xspan) return ROWOPS_ERR_INVALID_VALUE;
    return ROWOPS_OK;
}
}  // namespace

rowops_status_t rowops_row_sum(const void* x, float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                               cudaStream_t stream) {
    rowops_status_t st = check_reduce(x, out, M, N, ld, dtype);
    if (st != ROWOPS_OK || M == 0) return st;
    return reduce_dispatch(x, out, M, N, ld, dtype, 0, stream);
}

rowops_status_t rowops_row_max(const void* x, float* out, int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                               cudaStream_t stream) {
    rowops_status_t st = check_reduce(x, out, M, N, ld, dtype);
    if (st != ROWOPS_OK || M == 0) return st;
    return reduce_dispatch(x, out, M, N, ld, dtype, 1, stream);
}

rowops_status_t rowops_bias_residual_gelu(const void* x, const void* residual, const void* bias, void* y,
                                          int64_t M, int64_t N, int64_t ld, int approximate, rowops_dtype_t dtype,
                                          cudaStream_t stream) {
    if (approximate != 0 && approximate != 1) return ROWOPS_ERR_INVALID_VALUE;
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st == ROWOPS_OK && residual) st = check_rows(residual, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (M == 0) return ROWOPS_OK;
    const int es = elem_bytes(dtype);
    if (bias) {  // read by every row while y is written: apart from y's rows
        if (!aligned(bias, es)) return ROWOPS_ERR_INVALID_VALUE;
        const uintptr_t pb = reinterpret_cast<uintptr_t>(bias), py = reinterpret_cast<uintptr_t>(y);
        const uintptr_t sb = uintptr_t(N) * es, sy = uintptr_t(((M - 1) * ld + N) * es);
        if (pb < py + sy && py < pb + sb) return ROWOPS_ERR_INVALID_VALUE;
    }
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    const bool vec = tn.family != Family::Looped && N % (16 / es) == 0 && rows_aligned(x, y, ld, es) &&
                     (!residual || aligned(residual, 16)) && (!bias || aligned(bias, 16));
    const BiasResidualGeluLaunch fn = dtype == ROWOPS_F32 ? bias_residual_gelu_f32(approximate == 0, vec)
                                                          : bias_residual_gelu_bf16(approximate == 0, vec);
    return finish(fn(x, residual, bias, y, M, N, ld, cfg));
}

namespace {
rowops_status_t ln_gelu_dispatch(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                                 int64_t N, int64_t ld, rowops_dtype_t dtype, cudaStream_t stream, bool erf);
}  // namespace

rowops_status_t rowops_layernorm_gelu(const void* x, void* y, const void* w, const void* b,
                                      float eps, int64_t M, int64_t N, int64_t ld,
                                      rowops_dtype_t dtype, cudaStream_t stream) {
    return ln_gelu_dispatch(x, y, w, b, eps, M, N, ld, dtype, stream, false);
}

rowops_status_t rowops_layernorm_gelu_erf(const void* x, void* y, const void* w, const void* b, float eps,
                                          int64_t M, int64_t N, int64_t ld, rowops_dtype_t dtype,
                                          cudaStream_t stream) {
    return ln_gelu_dispatch(x, y, w, b, eps, M, N, ld, dtype, stream, true);
}

rowops_status_t rowops_gelu(const void* x, void* y, int64_t n, int approximate, rowops_dtype_t dtype,
                            cudaStream_t stream) {
    if (!valid_dtype(dtype) || n < 0 || (approximate != 0 && approximate != 1)) return ROWOPS_ERR_INVALID_VALUE;
    if (n == 0) return ROWOPS_OK;
    rowops_status_t st = check_rows(x, y, 1, n, n, dtype);  // one row of n elements
    if (st != ROWOPS_OK) return st;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    const GeluLaunch fn = dtype == ROWOPS_F32 ? gelu_f32(approximate == 0) : gelu_bf16(approximate == 0);
    return finish(fn(x, y, n, cfg));
}

namespace {
rowops_status_t ln_gelu_dispatch(const void* x, void* y, const void* w, const void* b, float eps, int64_t M,
                                 int64_t N, int64_t ld, rowops_dtype_t dtype, cudaStream_t stream, bool erf) {
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (!(eps >= 0.f) || eps == INFINITY) return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    const int es = elem_bytes(dtype);
    if ((w && !aligned(w, es)) || (b && !aligned(b, es))) return ROWOPS_ERR_INVALID_VALUE;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    // Short back-to-back rows by chunks of rows: those that are not whole
    // 16-byte vectors, those of at most 128 columns, and batches past 32 MiB
    // (where the row pipeline's per-row costs dominate). GB300, CUDA graphs,
    // 65536 rows, against the default before: bf16 N = 127 11.8 us (13.2), 33
    // 7.2 (13.0), 64 8.6 (12.5), 128 11.8 (12.6); fp32 N = 127 11.7 (13.9),
    // 255 20.9 (23.1), 256 21.0 (76.0). Aligned bf16 N = 200 and 256 stay
    // with the register rows (17.1 and 17.6 against 19.0 and 20.2).
    const bool short_rows = ld == N && N <= kFlatMaxN && aligned(x, 16) && aligned(y, 16);
    if (short_rows && (tn.family == Family::Flat ||
                       (tn.family == Family::Auto &&
                        ((N * es) % 16 != 0 || N <= 128 || big_batch(M, N, es))))) {
        if (const LnGeluLaunch fl = ln_gelu_flat(es, erf, N, tn.tpr))
            return finish(fl(x, y, w, b, eps, M, N, ld, cfg));
    }
    TmaChoice tc;
    if (pipeline_pays(tn, M, N, es, kPipeRowsNorm) &&
        choose_tma(x, y, N, ld, es, tn, {8, 4, 2, 3, 1}, &tc)) {
        const int tpr = kTmaBlocks[tc.block_index], vpt = kTmaVpts[tc.vpt_index];
        const int nbuf = ring_buffers(N, es, tma_affine_smem(tpr, vpt, es, tc.full, N), tn, cfg,
                                      tc.full ? 0 : size_t(tpr) * vpt * 16);
        if (nbuf > 0) {
            const TmaLnGeluLookup lookup = dtype == ROWOPS_F32 ? (erf ? ln_gelu_erf_tma_f32 : ln_gelu_tma_f32)
                                                               : (erf ? ln_gelu_erf_tma_bf16 : ln_gelu_tma_bf16);
            const int rows = choose_ln_rows(lookup, tpr, vpt, tc.full, N, nbuf, tn, cfg);
            const TmaLnGeluKernel k = lookup(tpr, vpt, rows, tc.full);
            if (k.launch) return finish(k.launch(x, y, w, b, eps, M, N, ld, nbuf, cfg));
        }
    }
    int tpr_index = 0, vpt = 0;
    LnGeluLaunch fn = nullptr;
    // static shared memory of the kernel (reduction buffers) stays under 256 bytes
    const bool smem_ok = ln_gelu_smem_bytes(N) + 256 <= size_t(cfg.max_smem_optin);
    if (tn.family != Family::Looped && smem_ok && same_phase(x, y) && choose_reg(N, es, tn, &tpr_index, &vpt)) {
        const bool al = rows_aligned(x, y, ld, es);
        fn = dtype == ROWOPS_F32 ? (erf ? ln_gelu_erf_reg_f32 : ln_gelu_reg_f32)(tpr_index, vpt, al)
                                 : (erf ? ln_gelu_erf_reg_bf16 : ln_gelu_reg_bf16)(tpr_index, vpt, al);
    }
    if (!fn)
        fn = dtype == ROWOPS_F32 ? (erf ? ln_gelu_erf_looped_f32 : ln_gelu_looped_f32)()
                                 : (erf ? ln_gelu_erf_looped_bf16 : ln_gelu_looped_bf16)();
    return finish(fn(x, y, w, b, eps, M, N, ld, cfg));
}
}  // namespace

rowops_status_t rowops_rmsnorm(const void* x, void* y, const void* w, float eps, int64_t M, int64_t N, int64_t ld,
                               rowops_dtype_t dtype, cudaStream_t stream) {
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (!(eps >= 0.f) || eps == INFINITY) return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    if (w && !aligned(w, elem_bytes(dtype))) return ROWOPS_ERR_INVALID_VALUE;
    return rms_dispatch(x, nullptr, y, nullptr, w, eps, M, N, ld, dtype, stream);
}

rowops_status_t rowops_fused_residual_rmsnorm(const void* x, const void* residual, void* y, void* residual_out,
                                              const void* w, float eps, int64_t M, int64_t N, int64_t ld,
                                              rowops_dtype_t dtype, cudaStream_t stream) {
    // each output either is one of the inputs or overlaps neither of them
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st == ROWOPS_OK) st = check_rows(residual, residual_out, M, N, ld, dtype);
    if (st == ROWOPS_OK) st = check_rows(x, residual_out, M, N, ld, dtype);
    if (st == ROWOPS_OK) st = check_rows(residual, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (!(eps >= 0.f) || eps == INFINITY) return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    const int es = elem_bytes(dtype);
    if (!rows_disjoint(y, residual_out, M, N, ld, es)) return ROWOPS_ERR_INVALID_VALUE;
    if (w && !aligned(w, es)) return ROWOPS_ERR_INVALID_VALUE;
    return rms_dispatch(x, residual, y, residual_out, w, eps, M, N, ld, dtype, stream);
}

size_t rowops_layernorm_gelu_backward_workspace_bytes(int64_t M, int64_t N, rowops_dtype_t dtype) {
    if (!valid_dtype(dtype) || M < 0 || N < 1 || N >= (int64_t(1) << 31)) return 0;
    // dw, db partials of at most bwd_max_partials(N) CTAs
    return size_t(bwd_max_partials(N)) * 2 * size_t(N) * sizeof(float);
}

rowops_status_t rowops_layernorm_gelu_backward(const void* x, const void* dy, const void* w, const void* b,
                                               float eps, void* dx, float* dw, float* db, int64_t M, int64_t N,
                                               int64_t ld, rowops_dtype_t dtype, void* workspace,
                                               size_t workspace_bytes, cudaStream_t stream) {
    rowops_status_t st = check_rows(x, dx, M, N, ld, dtype);
    if (st == ROWOPS_OK) st = check_rows(dy, dx, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (!(eps >= 0.f) || eps == INFINITY) return ROWOPS_ERR_INVALID_VALUE;
    const int es = elem_bytes(dtype);
    if ((w && !aligned(w, es)) || (b && !aligned(b, es))) return ROWOPS_ERR_INVALID_VALUE;
    if (!dw || !db || !aligned(dw, 4) || !aligned(db, 4)) return ROWOPS_ERR_INVALID_VALUE;
    {  // dw and db: N floats each, apart from each other
        const uintptr_t a = reinterpret_cast<uintptr_t>(dw), c = reinterpret_cast<uintptr_t>(db);
        const uintptr_t span = uintptr_t(N) * 4;
        if (a < c + span && c < a + span) return ROWOPS_ERR_INVALID_VALUE;
    }
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < rowops_layernorm_gelu_backward_workspace_bytes(M, N, dtype))
        return ROWOPS_ERR_WORKSPACE;
    {  // the partials are read while dw and db are written
        const uintptr_t ws = reinterpret_cast<uintptr_t>(workspace), span = uintptr_t(N) * 4;
        for (const float* o : {dw, db}) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(o);
            if (a < ws + workspace_bytes && ws < a + span) return ROWOPS_ERR_INVALID_VALUE;
        }
    }
    // dx is written while x and dy rows may still be read by other CTAs
    if (M > 0 && (!rows_disjoint(dx, x, M, N, ld, es) || !rows_disjoint(dx, dy, M, N, ld, es)))
        return ROWOPS_ERR_INVALID_VALUE;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    if (M == 0) {  // no rows: zero gradients
        if (cudaMemsetAsync(dw, 0, size_t(N) * 4, stream) != cudaSuccess ||
            cudaMemsetAsync(db, 0, size_t(N) * 4, stream) != cudaSuccess) {
            cudaGetLastError();
            return ROWOPS_ERR_CUDA;
        }
        return ROWOPS_OK;
    }
    float* part = static_cast<float*>(workspace);
    int grid = 0;
    cudaError_t e = cudaErrorUnknown;
    bool launched = false;
    // full rows on the row pipeline: x, dy, dx 16-byte aligned rows, a tile with
    // TPR * VPT = N / vec and at most 16 columns per thread
    const int64_t vec = 16 / es;
    const bool full = (tn.family == Family::Auto || tn.family == Family::Tma) && N % vec == 0 &&
                      rows_aligned(x, dx, ld, es) && aligned(dy, 16);
    if (full && tn.bwd != 1 && !tn.tpr && !tn.vpt) {
        // the dw, db partials in tensor memory: 512 threads as two row groups of
        // 256 (or four of 128) with TPR * VPT = N / vec, two ring slots per group,
        // every group's partials within the workspace's partial slots
        const int64_t nvec = N / vec;
        for (int tpr : {256, 128}) {
            if (launched || nvec % tpr) continue;
            const int vpt = int(nvec / tpr);
            const TmaBwdLaunch f = dtype == ROWOPS_F32 ? ln_gelu_bwd_tmem_f32(tpr, vpt) : ln_gelu_bwd_tmem_bf16(tpr, vpt);
            const int rows = 512 / tpr;
            const int nbuf = tn.ring >= 2 && tn.ring <= 4 ? tn.ring : 2;
            const size_t smem = size_t(kTmaRingHeader) + size_t(rows) * nbuf * 2 * tma_row_bytes(N, es) +
                                size_t(2) * vpt * tpr * vec * 4 + 1024;
            if (!f || smem > size_t(cfg.max_smem_optin) || bwd_max_partials(N) / rows < cfg.num_sms) continue;
            e = f(x, dy, w, b, eps, dx, part, M, N, ld, nbuf, &grid, cfg);
            launched = true;
        }
    }
    if (full && !launched) {
        const int64_t nvec = N / vec;
        // a tile: TPR * VPT = N / vec; the three-stage pipeline where 4..6 ring
        // slots fit (it holds three rows and wants one more in flight; or
        // ROWOPS_RING_BUFFERS), else one row at a time on 2 slots
        auto plan = [&](int ti, int vpt) -> bool {
            const size_t affine = size_t(2) * vpt * kBwdTpr[ti] * vec * 4;
            auto fits = [&](int nb) {
                return size_t(kTmaRingHeader) + size_t(nb) * 2 * tma_row_bytes(N, es) + affine + 1024 <=
                       size_t(cfg.max_smem_optin);
            };
            int nbuf = tn.ring > 0 ? (tn.ring > kTmaMaxSlots ? kTmaMaxSlots : tn.ring) : 6;
            while (nbuf > 4 && !fits(nbuf)) --nbuf;
            const bool pipe = nbuf >= 4 && fits(nbuf);
            if (!pipe) nbuf = 2;
            const TmaBwdLaunch f =
                dtype == ROWOPS_F32 ? ln_gelu_bwd_tma_f32(ti, vpt, pipe) : ln_gelu_bwd_tma_bf16(ti, vpt, pipe);
            if (!f || !fits(nbuf)) return false;
            e = f(x, dy, w, b, eps, dx, part, M, N, ld, nbuf, &grid, cfg);
            return true;
        };
        for (int v : {2, 4, 3, 1}) {
            if (launched) break;
            if (v * vec > 16 || nvec % v || (tn.vpt && tn.vpt != v)) continue;
            for (int i = 0; i < 5 && !launched; ++i)
                if (kBwdTpr[i] == nvec / v && (!tn.tpr || tn.tpr == kBwdTpr[i])) launched = plan(i, v);
        }
    }
    if (!launched) {
        const BwdLaunch f = dtype == ROWOPS_F32 ? ln_gelu_bwd_looped_f32() : ln_gelu_bwd_looped_bf16();
        e = f(x, dy, w, b, eps, dx, part, M, N, ld, &grid, cfg);
    }
    if (e != cudaSuccess) return finish(e);
    return finish(ln_gelu_bwd_reduce(part, grid, N, dw, db, cfg));
}

size_t rowops_online_softmax_workspace_bytes(int64_t M, int64_t N, rowops_dtype_t dtype) {
    if (!valid_dtype(dtype) || M < 0 || N < 1 || N >= (int64_t(1) << 31)) return 0;
    // the larger of the two forms' needs: the single-read form's header, M row
    // results and M * (ceil(N / 256) + 2) partial slots cover the two-launch
    // form's header and M * ceil(N / 256) partials
    const int64_t slots = persistent_slots(N);
    if (M > 0 && slots > (INT64_MAX / 16) / M) return 0;
    return size_t(256) + persistent_rowstat_bytes(M) + size_t(M) * size_t(slots) * 8u;
}

rowops_status_t rowops_online_softmax(const void* x, void* y, int64_t M, int64_t N, int64_t ld,
                                      rowops_dtype_t dtype, void* workspace,
                                      size_t workspace_bytes, int64_t chunk,
                                      cudaStream_t stream) {
    rowops_status_t st = check_rows(x, y, M, N, ld, dtype);
    if (st != ROWOPS_OK) return st;
    if (chunk != 0 && (chunk < kMinChunk || chunk > (int64_t(1) << 30) || chunk % 16 != 0))
        return ROWOPS_ERR_INVALID_VALUE;
    if (M == 0) return ROWOPS_OK;
    if (!workspace || !aligned(workspace, 256) ||
        workspace_bytes < rowops_online_softmax_workspace_bytes(M, N, dtype))
        return ROWOPS_ERR_WORKSPACE;
    const Tuning tn = tuning();
    LaunchCfg cfg;
    if ((st = make_cfg(stream, tn, &cfg)) != ROWOPS_OK) return st;
    const int es = elem_bytes(dtype);
    // The single-read forms (x read once; see online_softmax_persistent.cuh).
    // Row groups (each row spread over a group of CTAs that exchange slice
    // partials) are the default for batches above 32 MiB of rows of at least
    // 256 KiB: on GB300, 64 x 2^20 fp32 takes 101 us against 125 for the
    // two-launch form (and 104 against 133.5 between other row kernels).
    // Column slices of every row per CTA (`single_read`) only on request: no
    // faster than the two-launch form there.
    const bool groups_auto = tn.online == 0 && tn.family == Family::Auto &&
                             M * N * es > (int64_t(32) << 20) && N * es >= (int64_t(256) << 10);
    if (chunk == 0 && (tn.online == 3 || groups_auto) && rows_aligned(x, y, ld, es)) {
        GroupedLaunch gf = dtype == ROWOPS_F32 ? split_grouped_f32() : split_grouped_bf16();
        const cudaError_t e = gf(x, y, M, N, ld, workspace, tn.ring, cfg);
        if (e == cudaSuccess) return ROWOPS_OK;
        cudaGetLastError();
        // a grid the device will not co-schedule falls back to the two-launch form
        if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge) return ROWOPS_ERR_CUDA;
    }
    if (chunk == 0 && tn.online == 2 && rows_aligned(x, y, ld, es)) {
        PersistLaunch pf = dtype == ROWOPS_F32 ? split_persistent_f32() : split_persistent_bf16();
        const cudaError_t e = pf(x, y, M, N, ld, workspace, cfg);
        if (e == cudaSuccess) return ROWOPS_OK;
        cudaGetLastError();
        // a grid the device will not co-schedule falls back to the two-launch form
        if (e != cudaErrorNotSupported && e != cudaErrorCooperativeLaunchTooLarge) return ROWOPS_ERR_CUDA;
    }
    const int64_t n16 = (N + 15) / 16 * 16;
    if (chunk == 0) {
        // one unrolled step of a CTA per chunk, smaller while there are fewer
        // than four chunks per SM, never below the minimum
        chunk = split_step_cols(es);
        while (chunk > kMinChunk && M * ((N + chunk - 1) / chunk) < int64_t(4) * cfg.num_sms) chunk /= 2;
    }
    if (chunk > n16) chunk = n16 < kMinChunk ? kMinChunk : n16;
    const int64_t nchunks = (N + chunk - 1) / chunk;
    // chunks that are whole row-pipeline tiles of aligned rows stream through a
    // shared-memory ring (ROWOPS_RING_BUFFERS slots, default 3)
    if ((tn.family == Family::Auto || tn.family == Family::Tma) && rows_aligned(x, y, ld, es)) {
        const int nbuf = tn.ring > 0 ? (tn.ring > kTmaMaxSlots ? kTmaMaxSlots : tn.ring) : 3;
        const SplitTmaLaunch ft = dtype == ROWOPS_F32 ? split_softmax_tma_f32() : split_softmax_tma_bf16();
        const cudaError_t e = ft(x, y, M, N, ld, chunk, nchunks, nbuf, workspace, cfg);
        if (e != cudaErrorNotSupported) return finish(e);
    }
    SplitLaunch fn = dtype == ROWOPS_F32 ? split_softmax_f32() : split_softmax_bf16();
    return finish(fn(x, y, M, N, ld, chunk, nchunks, workspace, cfg));
}

rowops_status_t rowops_device_status(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return finish(cudaErrorUnknown);
    DeviceInfo di;
    if (device_info(dev, &di) != cudaSuccess) return finish(cudaErrorUnknown);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return finish(cudaErrorUnknown);
    unsigned word = 0;
    if (cudaMemcpy(&word, di.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return finish(cudaErrorUnknown);
    if (word != 0u) {
        const unsigned zero = 0u;
        if (cudaMemcpy(di.err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return finish(cudaErrorUnknown);
    }
    if (word == 0u) return ROWOPS_OK;
    return word == unsigned(ROWOPS_ERR_TIMEOUT) ? ROWOPS_ERR_TIMEOUT : ROWOPS_ERR_CUDA;
}

rowops_status_t rowops_online_softmax_status(const void* workspace, cudaStream_t stream) {
    if (!workspace) return ROWOPS_ERR_WORKSPACE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return finish(cudaErrorUnknown);
    unsigned word = 0;
    if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return finish(cudaErrorUnknown);
    if (word == 0u) return ROWOPS_OK;
    return word == unsigned(ROWOPS_ERR_TIMEOUT) ? ROWOPS_ERR_TIMEOUT : ROWOPS_ERR_CUDA;
}

}  // extern "C"
