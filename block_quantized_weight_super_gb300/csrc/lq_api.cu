// lq_api.cu -- the C ABI (include/lq.h): argument validation, launch
// planning and dispatch to the kernels.  Host code only, apart from the
// device status word.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/lq.h"
#include "lq_codec.cuh"
#include "lq_gv.cuh"
#include "lq_internal.h"

namespace lq {

// Status word the kernels set when a bounded wait runs out; its device
// address is passed to kernels (no relocatable device code needed).
static __device__ unsigned g_status_word = 0;


namespace {

thread_local char g_err[512] = "";
std::atomic<uint64_t> g_timeout_ns{1000000000ull};

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(LQ_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool fmt_ok(int fmt) { return fmt == FMT_Q4_K || fmt == FMT_Q6_K || fmt == FMT_Q8_0; }

int64_t rowbytes(int fmt, int64_t cols) { return cols / block_elems_of(fmt) * block_bytes_of(fmt); }

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Per-device facts and one-time set-up.
// Stages and partial-sum slots of the tensor-core kernel per cluster size
// (two CTAs per SM: at most 113 KB of shared memory each).
struct QmmCfg {
    int nstages, gmax;
};
QmmCfg qmm_cfg(int csize) { return csize >= 4 ? QmmCfg{2, 2} : QmmCfg{2, QMM_GROUP}; }

struct DevInfo {
    bool init = false;
    int sms = 0;
    unsigned* status = nullptr;
    int qmm_res[2][3] = {};       // resident tensor-core CTAs / clusters of 2 / of 4 (Q4_K, Q8_0)
    unsigned long long ctx = 0;   // id of the context these were taken in
    // scratch sets of the column-chunked batch-1 kernel, and the stream that
    // holds each (a set is bound to the first stream that needs it, for the
    // life of the context: launches on one stream run in order, so they can
    // share a set; launches on different streams must not)
    unsigned* gvw_cnt = nullptr;
    float* gvw_part = nullptr;
    cudaStream_t gvw_stream[GVW_SLOTS] = {};
    bool gvw_bound[GVW_SLOTS] = {};
};
std::mutex g_mu;
DevInfo g_dev[64];

}  // namespace

// Id of the current CUDA context (cuCtxGetId: unique for the life of the
// process, so a context created after cudaDeviceReset has a new one); 0 when
// no context is current.  Addresses of the library's device variables and
// per-function attributes belong to a context: caches keyed by this id are
// redone after a reset.  Without the driver entry points every context
// reads as 1 (caches are then never redone).
unsigned long long current_ctx_id() {
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static std::once_flag once;
    static GetCurrentFn get_cur = nullptr;
    static GetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess && a && b) {
            get_cur = reinterpret_cast<GetCurrentFn>(a);
            get_id = reinterpret_cast<GetIdFn>(b);
        }
    });
    if (!get_cur) return 1;
    CUcontext c = nullptr;
    if (get_cur(&c) != CUDA_SUCCESS || !c) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

namespace {

int dev_info(DevInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(LQ_EUNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo& d = g_dev[dev];
    const unsigned long long ctx = current_ctx_id();
    if (!d.init || ctx == 0 || ctx != d.ctx) {
        d.init = false;
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
        d.status = static_cast<unsigned*>(p);
        e = qmv1_set_smem(227 * 1024);
        if (e == cudaSuccess) e = qmv2_set_smem(227 * 1024);
        if (e == cudaSuccess) e = qmv4_set_smem(227 * 1024);
        if (e == cudaSuccess) e = qmv8_set_smem(227 * 1024);
        if (e == cudaSuccess) e = qmm_set_smem(FMT_Q4_K, 227 * 1024);
        if (e == cudaSuccess) e = qmm_set_smem(FMT_Q8_0, 227 * 1024);
        if (e == cudaSuccess) e = gv_set_smem(227 * 1024);
        if (e == cudaSuccess) e = gvw_scratch(&d.gvw_cnt, &d.gvw_part);
        for (int k = 0; k < GVW_SLOTS; ++k) {
            d.gvw_stream[k] = nullptr;
            d.gvw_bound[k] = false;
        }
        if (e == cudaSuccess) e = gemm_set_smem();
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        for (int f = 0; f < 2; ++f) {
            const int fmt = f ? FMT_Q8_0 : FMT_Q4_K;
            for (int i = 0, cs = 1; cs <= QMM_MAX_CSIZE; ++i, cs *= 2) {
                const QmmCfg q = qmm_cfg(cs);
                e = qmm_max_resident(fmt, cs, qmm_smem_bytes(fmt, q.nstages, cs, q.gmax), d.sms, &d.qmm_res[f][i]);
                if (e != cudaSuccess) return cuda_fail(e, "tensor-core matvec occupancy");
            }
        }
        d.ctx = current_ctx_id();     // the symbol lookup made the context current
        d.init = true;
    }
    *out = &d;
    return LQ_OK;
}

// ---------------------------------------------------------------- planning
struct QPlan {
    int B = 0, R = 0, NC = 0, RT = 0, ipt = 0, nstages = 0, stage_bytes = 0;
    size_t smem = 0;
};

// Geometry of the quantized matvec kernel for batch width B over `cols`
// with segments of the given formats.  Consumer threads NC*32 = U*m (U =
// cols/64 groups per row) so every thread takes the same number of work
// items (groups of R rows) from every tile of RT = R*m*j rows.  False if the
// kernel cannot take the shape (then the plain-load kernel is used).
int fmt_mask(const std::vector<int>& fmts) {
    int m = 0;
    for (int f : fmts) m |= f == FMT_Q4_K ? 1 : f == FMT_Q6_K ? 2 : 4;
    return (m == 5 || m == 6) ? 7 : m;
}

bool plan_qmv(int B, int64_t cols, const std::vector<int>& fmts, bool pairs, QPlan& p,
              int64_t rows = 0, int ctas = 0) {
    if (cols % 64 != 0 || cols <= 0 || cols > (1 << 20)) return false;
    const int64_t U = cols / 64;
    if (U > 512) return false;
    const int R = qmv_rows_per_item(B, fmt_mask(fmts));
    int64_t m = 1;
    while ((U * m) % 32) m *= 2;
    const int ncmax = qmv_max_consumer_warps(R);
    while (U * m / 32 < 4 && U * m / 32 * 2 <= ncmax) m *= 2;
    const int64_t NC = U * m / 32;
    if (NC > ncmax) return false;
    int64_t rbmax = 0;
    for (int f : fmts) rbmax = std::max<int64_t>(rbmax, rowbytes(f, cols));
    const int64_t unitrows = R * m;            // rows per tile step
    int64_t jmax = std::max<int64_t>(1, (32 * 1024) / (unitrows * rbmax));
    jmax = std::min<int64_t>(jmax, 8);
    // small matrices: keep at least `ctas` tiles so every CTA slot has work
    if (rows > 0 && ctas > 0) jmax = std::min<int64_t>(jmax, std::max<int64_t>(1, rows / (unitrows * ctas)));
    int64_t j = 0;
    for (int64_t jj = jmax; jj >= 1; --jj) {
        const int64_t RT = unitrows * jj;
        if (pairs && (RT & 1)) continue;
        bool aligned = true;
        for (int f : fmts)
            if (((pairs ? RT / 2 : RT) * rowbytes(f, cols)) % 16) aligned = false;
        if (j == 0) j = jj;
        if (aligned) {
            j = jj;
            break;
        }
    }
    if (j == 0) {
        if (!pairs) return false;
        j = 2;                                  // odd unitrows: two steps give an even tile
    }
    p.B = B;
    p.R = R;
    p.NC = (int)NC;
    p.ipt = (int)j;
    p.RT = (int)(unitrows * j);
    p.stage_bytes = (int)(((int64_t)p.RT * rbmax + 15) / 16 * 16 + 16);
    // Two stages: the producer copies them before waiting on the preceding
    // kernel, and more tiles requested at once delay the first one (measured
    // on GB300 in the decode layer: the Q6_K down 12.45 us with two stages,
    // 12.93 with up to six; no other workload changed).
    p.nstages = 2;
    p.smem = qmv_smem_bytes(B, (int)U, p.RT, p.nstages, p.stage_bytes);
    return p.smem <= 227 * 1024;
}

cudaError_t qmv_launch_b(int B, int mask, const QmvParams& P, int grid, int nt, size_t smem, cudaStream_t st) {
    return B == 1 ? qmv1_launch(mask, P, grid, nt, smem, st)
         : B == 2 ? qmv2_launch(mask, P, grid, nt, smem, st)
         : B == 4 ? qmv4_launch(mask, P, grid, nt, smem, st)
                  : qmv8_launch(mask, P, grid, nt, smem, st);
}

constexpr int GV_NOT_ELIGIBLE = -1;
constexpr int NEEDS_PREPASS = -2;

// A transform of the launch's x rows made before the matvec (GV_X_NORM:
// the RMS-norm of each row with weight nw and epsilon eps; GV_X_ACT: x rows
// of (g, u) pairs, the value act(g) * u).  The transformed rows
// ([batch][cols]) are written to `out` by whichever path runs.
struct XPre {
    int kind = GV_X_PLAIN;
    const float* nw = nullptr;
    float eps = 0.f;
    int act = ACT_NONE;
    float* out = nullptr;
};

// ---------------------------------------------------------------- launch plans
// Plans of recent launches, keyed by everything that shapes them: the
// segments (matrices, buffers, shapes, modes), cols, the batch width, the x
// transform and the context.  A decode loop repeats the same calls on the
// same buffers, and a plan (CTA partition, tile ring, occupancy) costs
// several microseconds of host time, more than the launch itself.  Keys are
// compared byte for byte (every key is zeroed before it is filled); on a hit
// only the wait limit and the status word are refreshed.
constexpr int PLAN_SEGS = 8;
constexpr int PLAN_ENTRIES = 512;          // a model's layers x calls per layer
struct PlanKey {
    unsigned long long ctx;
    int64_t cols;
    int32_t B, nseg, xkind, xact;
    float eps;
    int32_t pad;
    const float* xout;
    const float* xnw;
    Seg seg[PLAN_SEGS];
};
static_assert(sizeof(PlanKey) % 8 == 0, "plan keys are hashed as 64-bit words");

static bool plan_key(PlanKey& k, unsigned long long ctx, const std::vector<Seg>& segs, int64_t cols, int B,
                     const XPre* xp) {
    if (segs.size() > (size_t)PLAN_SEGS) return false;
    memset(&k, 0, sizeof k);
    k.ctx = ctx;
    k.cols = cols;
    k.B = B;
    k.nseg = (int32_t)segs.size();
    if (xp) {
        k.xkind = xp->kind;
        k.xact = xp->act;
        k.eps = xp->eps;
        k.xout = xp->out;
        k.xnw = xp->nw;
    } else {
        k.xkind = -1;
    }
    for (size_t i = 0; i < segs.size(); ++i) memcpy(&k.seg[i], &segs[i], sizeof(Seg));
    return true;
}

static uint64_t plan_hash(const PlanKey& k) {
    uint64_t w[sizeof(PlanKey) / 8];
    memcpy(w, &k, sizeof k);
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (uint64_t v : w) {
        h ^= v;
        h *= 0xBF58476D1CE4E5B9ull;
        h ^= h >> 31;
    }
    return h;
}

// A fixed ring of entries with a hash index; a hit is confirmed by
// comparing the whole key, and the oldest entry gives way to a new one.
template <class V>
struct PlanCache {
    std::mutex mu;
    std::vector<PlanKey> key;
    std::vector<V> val;
    std::vector<uint64_t> hash;
    std::unordered_map<uint64_t, int> index;
    int n = 0, next = 0;
    bool find(const PlanKey& k, V& v) {
        const uint64_t h = plan_hash(k);
        std::lock_guard<std::mutex> lk(mu);
        auto it = index.find(h);
        if (it == index.end() || memcmp(&key[it->second], &k, sizeof k) != 0) return false;
        v = val[it->second];
        return true;
    }
    void put(const PlanKey& k, const V& v) {
        const uint64_t h = plan_hash(k);
        std::lock_guard<std::mutex> lk(mu);
        if (key.empty()) {
            key.resize(PLAN_ENTRIES);
            val.resize(PLAN_ENTRIES);
            hash.resize(PLAN_ENTRIES);
        }
        if (n == PLAN_ENTRIES) {
            auto it = index.find(hash[next]);
            if (it != index.end() && it->second == next) index.erase(it);
        }
        key[next] = k;
        val[next] = v;
        hash[next] = h;
        index[h] = next;
        next = (next + 1) % PLAN_ENTRIES;
        n = std::min(n + 1, PLAN_ENTRIES);
    }
};

struct GvPlan {
    GvParams P;
    int mask, ncta;
    size_t smem;
};
struct QmvPlan {
    QmvParams P;
    int mask, B, grid, nt;
    size_t smem;
};
static PlanCache<GvPlan> g_gv_plans;
static PlanCache<QmvPlan> g_qmv_plans;

int run_gv(const std::vector<Seg>& segs, int64_t cols, cudaStream_t st, const XPre* pre);
int run_gvw(const std::vector<Seg>& segs, int64_t cols, cudaStream_t st, const XPre* pre);

// Run the segments (all sharing cols and the batch width B): at batch 1 the
// tensor-core kernel when it can take them, else the quantized matvec
// kernel when it can take the shape, else the plain-load kernel.  With a
// transform `pre`: fused where the chosen kernel has it (the batch-1
// tensor-core kernel: both; the quantized matvec kernel: the activation);
// otherwise NEEDS_PREPASS, before anything is launched.
int run_segments(std::vector<Seg>& segs, int B, int64_t cols, cudaStream_t st, const XPre* pre = nullptr) {
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    if (B == 1) {
        rc = run_gv(segs, cols, st, pre);
        if (rc != GV_NOT_ELIGIBLE) return rc;
    }
    if (B <= GVW_MAX_X) {
        rc = run_gvw(segs, cols, st, pre);
        if (rc != GV_NOT_ELIGIBLE) return rc;
    }
    if (pre && pre->kind == GV_X_NORM) return NEEDS_PREPASS;
    if (pre && pre->kind == GV_X_ACT) {
        if (!al(pre->out, 16)) return NEEDS_PREPASS;
        for (auto& s : segs) {
            s.xact = pre->act;
            s.xout = pre->out;
        }
    }
    PlanKey key;
    const bool keyed = plan_key(key, dev->ctx, segs, cols, B, nullptr);
    QmvPlan qp;
    if (keyed && g_qmv_plans.find(key, qp)) {
        qp.P.timeout_ns = g_timeout_ns.load();
        qp.P.status = dev->status;
        cudaError_t e = qmv_launch_b(qp.B, qp.mask, qp.P, qp.grid, qp.nt, qp.smem, st);
        return e == cudaSuccess ? LQ_OK : cuda_fail(e, "qmv launch");
    }
    // formats in order of first appearance (at most two per launch)
    std::vector<int> fmts;
    bool pairs = false;
    for (auto& s : segs) {
        if (std::find(fmts.begin(), fmts.end(), s.fmt) == fmts.end()) fmts.push_back(s.fmt);
        pairs = pairs || s.mode != MODE_PLAIN;
    }
    bool xal = true;                // the kernel stages x with 16-byte loads
    for (auto& s : segs) xal = xal && al(s.x, 16);
    int64_t rows = 0;               // matrix rows over all segments and batch chunks
    for (auto& s : segs) rows += (s.mode == MODE_PLAIN ? 1 : 2) * (int64_t)s.nout;
    QPlan pl;
    if (fmts.size() > 2 || !xal || !plan_qmv(B, cols, fmts, pairs, pl, rows, 2 * dev->sms)) {
        if (pre) return NEEDS_PREPASS;          // the plain-load kernel reads x as it is
        for (auto& s : segs) {
            if (s.nout <= 0) continue;
            cudaError_t e = launch_direct(s, cols, B, st);
            if (e != cudaSuccess) return cuda_fail(e, "direct matvec launch");
        }
        return LQ_OK;
    }
    // format group 0 segments first, then group 1
    std::vector<Seg> order;
    for (int f : fmts)
        for (auto& s : segs)
            if (s.fmt == f && s.nout > 0) order.push_back(s);
    const int nt = (pl.NC + 1) * 32;
    const int mask = fmt_mask(fmts);
    int per_sm = 0;
    cudaError_t e = B == 1 ? qmv1_occupancy(mask, nt, pl.smem, &per_sm)
                  : B == 2 ? qmv2_occupancy(mask, nt, pl.smem, &per_sm)
                  : B == 4 ? qmv4_occupancy(mask, nt, pl.smem, &per_sm)
                           : qmv8_occupancy(mask, nt, pl.smem, &per_sm);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy");
    if (per_sm < 1) per_sm = 1;
    for (size_t s0 = 0; s0 < order.size(); s0 += MAX_SEG) {
        QmvParams P;
        memset(&P, 0, sizeof P);
        int t = 0, n = 0, t0 = -1;
        P.fmt0 = P.fmt1 = order[s0].fmt;
        for (size_t i = s0; i < order.size() && i < s0 + MAX_SEG; ++i) {
            Seg s = order[i];
            if (s.fmt != P.fmt0 && t0 < 0) {
                t0 = t;
                P.fmt1 = s.fmt;
            }
            const int opt = s.mode == MODE_PLAIN ? pl.RT : pl.RT / 2;
            s.tile0 = t;
            s.ntiles = (s.nout + opt - 1) / opt;
            t += s.ntiles;
            P.seg[n++] = s;
        }
        P.nseg = n;
        P.ntiles = t;
        QGeo& G = P.geo;
        G.cols = (int32_t)cols;
        G.U = (int32_t)(cols / 64);
        G.UP = qmv_red_stride(G.U);
        G.RT = pl.RT;
        G.ipt = pl.ipt;
        for (int i = 0; i < n; ++i)
            if (P.seg[i].bcnt || P.seg[i].boff) P.dev_counts = 1;
        P.R = pl.R;
        P.nstages = pl.nstages;
        P.stage_bytes = pl.stage_bytes;
        P.timeout_ns = g_timeout_ns.load();
        P.status = dev->status;
        int grid = std::min(dev->sms * per_sm, t);
        if (t0 < 0) {
            P.tile_split = t;
            P.cta_split = grid;
        } else {
            if (grid < 2) grid = 2;
            P.tile_split = t0;
            int g0 = (int)((int64_t)grid * t0 / t);
            g0 = std::max(1, std::min(grid - 1, g0));
            P.cta_split = g0;
        }
        e = qmv_launch_b(B, mask, P, grid, nt, pl.smem, st);
        if (e != cudaSuccess) return cuda_fail(e, "qmv launch");
        if (keyed && order.size() <= (size_t)MAX_SEG) {
            qp.P = P;
            qp.mask = mask;
            qp.B = B;
            qp.grid = grid;
            qp.nt = nt;
            qp.smem = pl.smem;
            g_qmv_plans.put(key, qp);
        }
    }
    return LQ_OK;
}

// ---------------------------------------------------------------- tensor maps
// 2-D tensor maps over quantized matrices (uint32 elements, a matrix row per
// tensor row), encoded once per (base, rows, row bytes, stride, box rows)
// through the driver entry point and cached.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct MapKey {
    const void* base;
    int64_t rows, rowbytes, stride;
    int box_inner, box_rows;
    bool operator==(const MapKey& o) const {
        return base == o.base && rows == o.rows && rowbytes == o.rowbytes && stride == o.stride &&
               box_inner == o.box_inner && box_rows == o.box_rows;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        size_t h = std::hash<const void*>()(k.base);
        for (int64_t v : {k.rows, k.rowbytes, k.stride, (int64_t)k.box_inner, (int64_t)k.box_rows})
            h = h * 1000003u ^ std::hash<int64_t>()(v);
        return h;
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
EncodeTiledFn g_encode = nullptr;

// box: box_inner uint32 elements (a row's bytes of one tile) x box_rows rows
int tensor_map(CUtensorMap* out, const void* base, int64_t rows, int64_t rowbytes, int64_t stride, int box_inner,
               int box_rows) {
    const MapKey key{base, rows, rowbytes, stride, box_inner, box_rows};
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = it->second;
        return LQ_OK;
    }
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(LQ_ECUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)(rowbytes / 4), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap m;
    const CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(LQ_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    if (g_maps.size() >= 4096) g_maps.clear();
    g_maps.emplace(key, m);
    *out = m;
    return LQ_OK;
}


// ---------------------------------------------------------------- batch-1 tensor-core path
// Segments of one x row (no device counts or gathers), Q4_K alone or Q4_K
// with Q6_K, whose columns are a multiple of 256, with rows a multiple of 4
// bytes, weights 4-byte aligned and a 16-row tile of at most
// GV_MAX_TILE_BYTES.  Returns GV_NOT_ELIGIBLE otherwise: Q6_K alone and Q8_0
// run faster on the CUDA-core kernel at batch 1 (measured per launch on
// GB300: the down projection and the Q8_0 FFN).
//
// Plan: one CTA per SM; the row blocks are split into contiguous ranges of
// nearly equal weight bytes, one per CTA; tiles land in a ring of up to
// GV_MAX_INFLIGHT slots, as many as shared memory holds.
int run_gv(const std::vector<Seg>& segs, int64_t cols, cudaStream_t st, const XPre* xp) {
    if (segs.empty() || segs.size() > (size_t)GV_MAX_SEG || cols % 256 != 0 || cols > (1 << 20))
        return GV_NOT_ELIGIBLE;
    if (xp && xp->kind != GV_X_PLAIN && (!al(xp->out, 16) || (xp->kind == GV_X_NORM && !al(xp->nw, 16))))
        return GV_NOT_ELIGIBLE;
    int mask = 0;
    for (auto& s : segs) {
        if (s.nbatch != 1 || s.b0 != 0 || s.xmap || s.boff || s.bcnt || s.x != segs[0].x) return GV_NOT_ELIGIBLE;
        if (s.mode != MODE_PLAIN && s.mode != MODE_PAIR_INTERLEAVED) return GV_NOT_ELIGIBLE;
        if (s.fmt != FMT_Q4_K && s.fmt != FMT_Q6_K) return GV_NOT_ELIGIBLE;
        mask |= s.fmt == FMT_Q4_K ? 1 : 2;
    }
    if (!(mask & 1)) return GV_NOT_ELIGIBLE;
    // the kernel instances are gv_kernel<1> (Q4_K) and gv_kernel<3> (both
    // formats): the shared-memory layout is sized for the instance launched
    mask = mask == 1 ? 1 : 3;
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    PlanKey key;
    const bool keyed = plan_key(key, dev->ctx, segs, cols, 1, xp ? xp : nullptr);
    GvPlan gp;
    if (keyed && g_gv_plans.find(key, gp)) {
        gp.P.timeout_ns = g_timeout_ns.load();
        gp.P.status = dev->status;
        cudaError_t e = gv_launch(gp.mask, gp.P, gp.ncta, gp.smem, st);
        return e == cudaSuccess ? LQ_OK : cuda_fail(e, "batch-1 tensor-core matvec launch");
    }
    const int nsb = (int)(cols / 256);
    if (nsb > GV_MAX_NSB) return GV_NOT_ELIGIBLE;
    GvParams P;
    memset(&P, 0, sizeof P);
    std::vector<double> rbcost;            // weight bytes of a row block, in Q4_K super-blocks
    uint32_t slot = 0;
    int n = 0;
    for (auto& s : segs) {
        if (s.nout <= 0) continue;
        const bool pair = s.mode != MODE_PLAIN;
        const int64_t rb = rowbytes(s.fmt, cols);
        if (rb % 4 != 0 || !al(s.w, 4) || GV_ROWS * rb > GV_MAX_TILE_BYTES) return GV_NOT_ELIGIBLE;
        GvSeg& G = P.seg[n];
        G.w = s.w;
        G.y = s.y;
        G.rowbytes = rb;
        G.fmt = s.fmt;
        G.mode = s.mode;
        G.act = s.act;
        G.cap = s.cap;
        G.nout = s.nout;
        G.nrows = (pair ? 2 : 1) * s.nout;
        G.nrb = pair ? (s.nout + 7) / 8 : (s.nout + GV_ROWS - 1) / GV_ROWS;
        G.rb0 = (int32_t)rbcost.size();
        uint32_t bytes;
        if (al(s.w, 16) && (G.nrows * rb) % 16 == 0) {
            G.copy = GV_COPY_TILE;
            bytes = (uint32_t)(GV_ROWS * rb);
        } else {
            G.copy = GV_COPY_CPA;
            G.pitch = gv_row_pitch(s.fmt, nsb);
            bytes = (uint32_t)(GV_ROWS * G.pitch);
        }
        slot = std::max(slot, (bytes + 127u) & ~127u);
        const double c = gv_span(s.fmt) / 144.0;
        for (int i = 0; i < G.nrb; ++i) rbcost.push_back(c);
        ++n;
    }
    if (n == 0) return LQ_OK;
    const int nrb = (int)rbcost.size();
    std::vector<double> pre(nrb + 1, 0.0);
    for (int i = 0; i < nrb; ++i) pre[i + 1] = pre[i] + rbcost[i];
    const int ncta = std::min(std::min(dev->sms, GV_MAX_CTA), nrb);
    std::vector<int> b(ncta + 1, 0);
    b[ncta] = nrb;
    for (int k = 1; k < ncta; ++k) {
        const double target = pre[nrb] * k / ncta;
        int i = (int)(std::lower_bound(pre.begin(), pre.end(), target) - pre.begin());
        if (i > 0 && target - pre[i - 1] < pre[i] - target) --i;
        b[k] = std::max(b[k - 1] + 1, std::min(i, nrb - (ncta - k)));
    }
    int mxt = 0;
    for (int k = 0; k < ncta; ++k) mxt = std::max(mxt, b[k + 1] - b[k]);
    if (mxt > GV_MAX_TILES) return GV_NOT_ELIGIBLE;
    // a ring of up to GV_MAX_INFLIGHT tiles: enough bytes in flight per SM to
    // keep HBM busy, few enough that they land one after another and the
    // warps compute each as it arrives
    int ns = std::min(GV_MAX_INFLIGHT, std::max(2, mxt));
    while (ns >= 2 && gv_layout(mask, ns, slot, mxt, nsb, ns).total > GV_SMEM_MAX) --ns;
    if (ns < 2) return GV_NOT_ELIGIBLE;
    P.nseg = n;
    P.x = segs[0].x;
    P.timeout_ns = g_timeout_ns.load();
    P.status = dev->status;
    P.nsb = nsb;
    P.nslots = ns;
    P.slot_bytes = slot;
    P.maxtiles = mxt;
    P.x16 = al(segs[0].x, 16) ? 1 : 0;
    if (xp) {
        P.xpre = xp->kind;
        P.act = xp->act;
        P.nw = xp->nw;
        P.eps = xp->eps;
        P.xout = xp->kind != GV_X_PLAIN ? xp->out : nullptr;
    }
    for (int k = 0; k <= ncta; ++k) P.cta_rb[k] = b[k];
    const size_t smem = gv_layout(mask, ns, slot, mxt, nsb, ns).total;
    cudaError_t e = gv_launch(mask, P, ncta, smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "batch-1 tensor-core matvec launch");
    if (keyed) {
        gp.P = P;
        gp.mask = mask;
        gp.ncta = ncta;
        gp.smem = smem;
        g_gv_plans.put(key, gp);
    }
    return LQ_OK;
}

// The scratch set of stream st for the column-chunked kernel: the set bound
// to st, else a free one (bound now); -1 when every set is bound to another
// stream.
static int gvw_slot(DevInfo* dev, cudaStream_t st) {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int k = 0; k < GVW_SLOTS; ++k)
        if (dev->gvw_bound[k] && dev->gvw_stream[k] == st) return k;
    for (int k = 0; k < GVW_SLOTS; ++k)
        if (!dev->gvw_bound[k]) {
            dev->gvw_bound[k] = true;
            dev->gvw_stream[k] = st;
            return k;
        }
    return -1;
}

struct GvwPlan {
    GvwParams P;
    int fmt = 0, nm = 1, ncta = 0;
    size_t smem = 0;
};
static PlanCache<GvwPlan> g_gvw_plans;

// One plain Q4_K or Q6_K matrix at batch 1 that the whole-row kernel does not
// take (rows too wide for a tile, or Q6_K alone), or a Q6_K matrix against 2
// to 8 plain x rows, on the column-chunked kernel: items of 16 rows x ch
// super-blocks (ch = 7 for Q4_K, 8 for Q6_K: a row piece of 1008 or 1680
// bytes, an odd multiple of 16, so the rows a quarter-warp reads fall in
// distinct banks), spread evenly over one CTA per SM in column-major order.
// Needs W 16-byte aligned with rows a multiple of 16 bytes (every row piece
// one bulk copy) and no input norm (it needs whole rows).
int run_gvw(const std::vector<Seg>& segs, int64_t cols, cudaStream_t st, const XPre* xp) {
    if (segs.size() != 1 || cols % 256 != 0 || cols > (1 << 20)) return GV_NOT_ELIGIBLE;
    const Seg& s = segs[0];
    const int M = s.nbatch;
    if (M < 1 || M > GVW_MAX_X || s.xmap || s.boff || s.bcnt || s.mode != MODE_PLAIN) return GV_NOT_ELIGIBLE;
    if (s.fmt != FMT_Q4_K && s.fmt != FMT_Q6_K) return GV_NOT_ELIGIBLE;
    if (M > 1 && (s.fmt != FMT_Q6_K || (xp && xp->kind != GV_X_PLAIN))) return GV_NOT_ELIGIBLE;
    if (xp && (xp->kind == GV_X_NORM || (xp->kind == GV_X_ACT && !al(xp->out, 16)))) return GV_NOT_ELIGIBLE;
    const int nm = M == 1 ? 1 : M <= 4 ? 4 : 8;           // the kernel instance's x rows
    const int64_t rb = rowbytes(s.fmt, cols);
    if (!al(s.w, 16) || rb % 16 != 0 || s.nout <= 0) return GV_NOT_ELIGIBLE;
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    PlanKey key;
    const bool keyed = plan_key(key, dev->ctx, segs, cols, M, xp ? xp : nullptr);
    GvwPlan gp;
    const bool cached = keyed && g_gvw_plans.find(key, gp);
    if (!cached) {
        const int span = s.fmt == FMT_Q4_K ? 144 : 210;
        const int ch = s.fmt == FMT_Q4_K ? 7 : 8;
        const int nsb = (int)(cols / 256);
        const int nch = (nsb + ch - 1) / ch;
        const int64_t nrb = (s.nout + GV_ROWS - 1) / GV_ROWS;
        // several x rows pay off against the CUDA-core kernel from 3 rows of
        // several chunks (Q6_K 2560 x 10240: 8 rows 38.4 us against 62.4, 5
        // rows 33.4 against 46.6, 2 rows 18.3 against 18.6; 1024 x 2048, one
        // chunk, 8 rows: 10.5 against 8.6)
        if (M > 1 && (M < 3 || nch < 2)) return GV_NOT_ELIGIBLE;
        // with many row blocks the CUDA-core kernel's row partition is even
        // already and the cross-CTA chunk sums only cost (measured: Q4_K
        // 14336 x 8192, 5.9 row blocks per SM, 28.2 us here against 27.3)
        if (nch > 1 && nrb >= (int64_t)GVW_MAX_RB_PER_SM * dev->sms) return GV_NOT_ELIGIBLE;
        if (nch > 1 && (nrb > GVW_MAX_RB || (int64_t)nch * nrb * GV_ROWS * nm > GVW_MAX_PART)) return GV_NOT_ELIGIBLE;
        const int64_t nitems = (int64_t)nch * nrb;
        if (nitems > (int64_t)GV_MAX_TILES * GV_MAX_CTA) return GV_NOT_ELIGIBLE;
        const int ncta = (int)std::min<int64_t>(std::min(dev->sms, GV_MAX_CTA), nitems);
        GvwParams& P = gp.P;
        memset(&P, 0, sizeof P);
        int maxtiles = 0, winsb = 0;
        for (int k = 0; k <= ncta; ++k) P.cta_j[k] = (int32_t)(nitems * k / ncta);
        for (int k = 0; k < ncta; ++k) {
            const int64_t jA = P.cta_j[k], jB = P.cta_j[k + 1];
            maxtiles = std::max(maxtiles, (int)(jB - jA));
            const int cA = (int)(jA / nrb), cB = (int)((jB - 1) / nrb);
            winsb = std::max(winsb, std::min(nsb, (cB + 1) * ch) - cA * ch);
        }
        if (maxtiles > GV_MAX_TILES || winsb > GV_MAX_NSB) return GV_NOT_ELIGIBLE;
        const uint32_t slot = ((uint32_t)(GV_ROWS * ch * span) + 127u) & ~127u;
        int ns = std::min(GV_MAX_INFLIGHT, std::max(2, maxtiles));
        while (ns >= 2 && gvw_smem_bytes(nm, ns, slot, maxtiles, winsb, ch) > GV_SMEM_MAX) --ns;
        if (ns < 2) return GV_NOT_ELIGIBLE;
        P.w = s.w;
        P.y = s.y + (int64_t)s.b0 * s.ld_y;
        P.x = s.x + (int64_t)s.b0 * cols;
        P.nx = M;
        P.ld_x = cols;
        P.ld_y = s.ld_y;
        P.rowbytes = rb;
        P.rows = s.nout;
        P.nsb = nsb;
        P.ch = ch;
        P.nch = nch;
        P.nrb = (int32_t)nrb;
        P.pitch = ch * span;
        P.slot_bytes = slot;
        P.nslots = ns;
        P.maxtiles = maxtiles;
        P.winsb = winsb;
        P.x16 = al(P.x, 16) ? 1 : 0;
        P.cap = s.cap;
        if (xp) {
            P.xpre = xp->kind;
            P.act = xp->act;
            P.xout = xp->kind != GV_X_PLAIN ? xp->out : nullptr;
        }
        gp.fmt = s.fmt;
        gp.nm = nm;
        gp.ncta = ncta;
        gp.smem = gvw_smem_bytes(nm, ns, slot, maxtiles, winsb, ch);
    }
    GvwParams P = gp.P;
    if (P.nch > 1) {
        const int k = gvw_slot(dev, st);
        if (k < 0) return GV_NOT_ELIGIBLE;
        P.cnt = dev->gvw_cnt + (size_t)k * GVW_MAX_RB;
        P.part = dev->gvw_part + (size_t)k * GVW_MAX_PART;
    }
    P.timeout_ns = g_timeout_ns.load();
    P.status = dev->status;
    cudaError_t e = gvw_launch(gp.fmt, gp.nm, P, gp.ncta, gp.smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "column-chunked tensor-core matvec launch");
    if (keyed && !cached) g_gvw_plans.put(key, gp);
    return LQ_OK;
}

// ---------------------------------------------------------------- tensor-core path
// Q4_K or Q8_0 segments (one format) of up to QMM_NT x rows whose columns
// are a multiple of the tile width, with 16-byte aligned weights and x
// (tensor maps, bulk copies).
bool qmm_eligible(const std::vector<Seg>& segs, int64_t cols) {
    if (segs.empty() || !qmm_format_ok(segs[0].fmt)) return false;
    if (cols % qmm_kc(segs[0].fmt) != 0 || cols > (1 << 20)) return false;
    for (auto& s : segs) {
        if (s.fmt != segs[0].fmt) return false;
        if (!al(s.w, 16) || (s.w2 && !al(s.w2, 16)) || !al(s.x, 16)) return false;
    }
    return true;
}

// Run segments on the tensor-core kernel.  Row blocks are QMM_RT weight rows
// (pairs count twice); a cluster of csize CTAs splits a row block's column
// chunks when there are too few row blocks to fill the resident CTAs.
int run_qmm(std::vector<Seg>& segs, int64_t cols, cudaStream_t st) {
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    const int fmt = segs[0].fmt;
    const int f = fmt == FMT_Q8_0 ? 1 : 0;
    const int nchunk = (int)(cols / qmm_kc(fmt));
    const int box_inner = qmm_wrow(fmt) / 4;
    auto blocks_of = [](const Seg& s) {
        const int64_t r = (s.mode == MODE_PLAIN ? 1 : 2) * (int64_t)s.nout;
        return (r + QMM_RT - 1) / QMM_RT;
    };
    int64_t nb_all = 0;
    for (auto& s : segs) nb_all += blocks_of(s);
    if (nb_all == 0) return LQ_OK;
    // cluster size: fewest (rounds of row blocks) x (chunks per CTA), a small
    // charge per extra rank for the partial-sum exchange
    int ci = 0;
    double best = 0.0;
    for (int i = 0, cs = 1; cs <= QMM_MAX_CSIZE && cs <= nchunk; ++i, cs *= 2) {
        const int res = dev->qmm_res[f][i];
        if (res < 1) continue;
        const double t = (double)((nb_all + res - 1) / res) * ((nchunk + cs - 1) / cs) * (1.0 + 0.05 * (cs - 1));
        if (best == 0.0 || t < best) {
            best = t;
            ci = i;
        }
    }
    const int cs = 1 << ci, res = std::max(1, dev->qmm_res[f][ci]);
    const QmmCfg qc = qmm_cfg(cs);
    const size_t smem = qmm_smem_bytes(fmt, qc.nstages, cs, qc.gmax);
    const int64_t rb = rowbytes(fmt, cols);
    for (size_t s0 = 0; s0 < segs.size(); s0 += QMM_MAX_SEG) {
        QmmParams P;
        memset(&P, 0, sizeof P);
        int t = 0, n = 0;
        for (size_t i = s0; i < segs.size() && i < s0 + QMM_MAX_SEG; ++i) {
            Seg s = segs[i];
            s.tile0 = t;
            s.ntiles = (int32_t)blocks_of(s);
            t += s.ntiles;
            if (s.mode == MODE_PLAIN) {
                rc = tensor_map(&P.tm[n][0], s.w, s.nout, rb, rb, box_inner, QMM_RT);
            } else if (s.mode == MODE_PAIR_TWO) {
                rc = tensor_map(&P.tm[n][0], s.w, s.nout, rb, rb, box_inner, QMM_PAIR_BOX);
                if (!rc) rc = tensor_map(&P.tm[n][1], s.w2, s.nout, rb, rb, box_inner, QMM_PAIR_BOX);
            } else {                        // packed gate / up: rows 2i and 2i + 1
                rc = tensor_map(&P.tm[n][0], s.w, s.nout, rb, 2 * rb, box_inner, QMM_PAIR_BOX);
                if (!rc) rc = tensor_map(&P.tm[n][1], s.w + rb, s.nout, rb, 2 * rb, box_inner, QMM_PAIR_BOX);
            }
            if (rc) return rc;
            P.seg[n++] = s;
        }
        if (t == 0) continue;
        P.nseg = n;
        P.nblocks = t;
        P.cols = (int32_t)cols;
        P.nchunk = nchunk;
        // units of gmax row blocks, dealt round robin to the clusters: as
        // large as the slots allow while every cluster still gets one
        const int ncl0 = std::min(res, t);
        const int gmax = std::max(1, std::min(qc.gmax, (t + ncl0 - 1) / ncl0));
        const int ncl = std::min(res, (t + gmax - 1) / gmax);
        P.nstages = qc.nstages;
        P.csize = cs;
        P.gmax = gmax;
        for (int i = 0; i < n; ++i)
            if (P.seg[i].bcnt || P.seg[i].boff) P.dev_counts = 1;
        P.timeout_ns = g_timeout_ns.load();
        P.status = dev->status;
        const int grid = cs * ncl;
        cudaError_t e = qmm_launch(fmt, P, grid, smem, st);
        if (e != cudaSuccess) return cuda_fail(e, "tensor-core matvec launch");
    }
    return LQ_OK;
}

// Batch from which a dense call takes the tensor-core kernel (never for
// formats it does not handle).
int qmm_min_batch(int fmt) {
    return fmt == FMT_Q4_K ? QMM_MIN_BATCH : fmt == FMT_Q8_0 ? QMM_MIN_BATCH_Q8 : 1 << 30;
}

// Widest batch width (4, 2 or 1) the quantized matvec kernel can plan for
// these columns and formats (x for B rows must fit in shared memory).
// x rows per pass of the quantized matvec kernel: 8 for batches of 5 or
// more (the weights read once for up to 8 rows), 4 for 3 or 4, else the
// batch; narrower when the plan does not fit (x staged for B rows).
int batch_width(int64_t cols, int batch, const std::vector<int>& fmts, bool pairs) {
    int B = batch >= 5 ? 8 : batch >= 3 ? 4 : batch;
    QPlan pl;
    while (B > 1 && !plan_qmv(B, cols, fmts, pairs, pl)) B /= 2;
    return B;
}

Seg plain_seg(int fmt, const void* W, int64_t rows, const float* x, float* y, int64_t ld_y, int b0,
              int nb) {
    Seg s;
    memset(&s, 0, sizeof s);
    s.w = static_cast<const uint8_t*>(W);
    s.x = x;
    s.y = y;
    s.ld_y = ld_y;
    s.nout = (int32_t)rows;
    s.fmt = fmt;
    s.mode = MODE_PLAIN;
    s.b0 = b0;
    s.nbatch = nb;
    return s;
}

int check_mat(int fmt, const void* W, int64_t rows, int64_t cols, const char* name) {
    if (!fmt_ok(fmt)) return fail(LQ_EINVAL, "%s: unknown format %d", name, fmt);
    if (rows < 0 || cols <= 0) return fail(LQ_ESHAPE, "%s: rows %lld cols %lld", name, (long long)rows, (long long)cols);
    if (cols % block_elems_of(fmt) != 0)
        return fail(LQ_ESHAPE, "%s: cols %lld not a multiple of %d", name, (long long)cols, block_elems_of(fmt));
    if (rows > (int64_t)1 << 30 || cols > (int64_t)1 << 20)
        return fail(LQ_ESHAPE, "%s: size out of range", name);
    if (rows > 0 && !W) return fail(LQ_EINVAL, "%s: null weights", name);
    if (W && !al(W, 2)) return fail(LQ_EALIGN, "%s: weights not 2-byte aligned", name);
    return LQ_OK;
}

int check_f32(const void* p, const char* name) {
    if (!p) return fail(LQ_EINVAL, "%s is null", name);
    if (!al(p, 4)) return fail(LQ_EALIGN, "%s not 4-byte aligned", name);
    return LQ_OK;
}

// Everything lq_moe_ffn_ex checks before it looks at the workspace.
int moe_validate(const float* router, int E, int topk, int norm, int fmt, const void* const* W1,
                 const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter, int n_shared,
                 const void* const* Ws1, const void* const* Ws3, const void* const* Ws2, int64_t inter_s,
                 const float* shared_gate, const float* X, float* Y, int ntok, int32_t* topk_idx,
                 float* topk_w) {
    if (E < 1 || E > 256) return fail(LQ_EINVAL, "n_experts %d", E);
    if (topk < 1 || topk > E) return fail(LQ_EINVAL, "topk %d with %d experts", topk, E);
    if (norm != 0 && norm != 1) return fail(LQ_EINVAL, "norm_topk_prob %d", norm);
    if (ntok < 0) return fail(LQ_EINVAL, "ntok %d", ntok);
    if (n_shared < 0 || n_shared > LQ_MOE_MAX_SHARED) return fail(LQ_EINVAL, "n_shared %d", n_shared);
    if (!W1 || !W3 || !W2) return fail(LQ_EINVAL, "expert pointer arrays are null");
    int rc;
    for (int e = 0; e < E; ++e) {
        if ((rc = check_mat(fmt, W1[e], inter, hidden, "W1")) || (rc = check_mat(fmt, W3[e], inter, hidden, "W3")) ||
            (rc = check_mat(fmt, W2[e], hidden, inter, "W2")))
            return rc;
        if (!W1[e] || !W3[e] || !W2[e]) return fail(LQ_EINVAL, "expert %d weights null", e);
    }
    if (n_shared > 0) {
        if (!Ws1 || !Ws3 || !Ws2) return fail(LQ_EINVAL, "shared-expert pointer arrays are null");
        for (int e = 0; e < n_shared; ++e) {
            if ((rc = check_mat(fmt, Ws1[e], inter_s, hidden, "Ws1")) ||
                (rc = check_mat(fmt, Ws3[e], inter_s, hidden, "Ws3")) ||
                (rc = check_mat(fmt, Ws2[e], hidden, inter_s, "Ws2")))
                return rc;
            if (!Ws1[e] || !Ws3[e] || !Ws2[e]) return fail(LQ_EINVAL, "shared expert %d weights null", e);
        }
    } else if (shared_gate) {
        return fail(LQ_EINVAL, "shared_gate given without shared experts");
    }
    if (ntok == 0) return LQ_OK;
    if ((long long)ntok * E * 4 > 48 * 1024) return fail(LQ_ESHAPE, "ntok * n_experts too large");
    if ((rc = check_f32(router, "router")) || (rc = check_f32(X, "X")) || (rc = check_f32(Y, "Y"))) return rc;
    if (shared_gate && (rc = check_f32(shared_gate, "shared_gate"))) return rc;
    if ((topk_idx && !al(topk_idx, 4)) || (topk_w && !al(topk_w, 4)))
        return fail(LQ_EALIGN, "topk outputs not 4-byte aligned");
    return LQ_OK;
}

// The tensor-core kernel takes the grouped launches when every matrix of
// the launch has a tile-multiple width and 16-byte aligned rows.
bool moe_tc_ok(int fmt, int ntok, int64_t hidden, int64_t inter, const void* const* W1, const void* const* W3,
               const void* const* W2, int n, const float* X) {
    bool tc = ntok >= QMM_MOE_MIN_TOKENS && qmm_format_ok(fmt) && hidden % qmm_kc(fmt) == 0 &&
              inter % qmm_kc(fmt) == 0 && al(X, 16);
    for (int ex = 0; tc && ex < n; ++ex) tc = al(W1[ex], 16) && al(W3[ex], 16) && al(W2[ex], 16);
    return tc;
}

}  // namespace
}  // namespace lq

using namespace lq;

// Scratch of lq_moe_ffn_static: a file-scope device array (no allocation),
// one instance per device.
static __device__ __align__(256) uint8_t g_moe_scratch[LQ_MOE_STATIC_SCRATCH_BYTES];
constexpr int kMaxDevices = 64;
static std::mutex g_moe_scratch_mu;
static void* g_moe_scratch_ptr[kMaxDevices] = {};
static unsigned long long g_moe_scratch_ctx[kMaxDevices] = {};

extern "C" {

size_t lq_block_bytes(int fmt) { return fmt_ok(fmt) ? (size_t)block_bytes_of(fmt) : 0; }
int lq_block_elems(int fmt) { return fmt_ok(fmt) ? block_elems_of(fmt) : 0; }
int64_t lq_row_bytes(int fmt, int64_t cols) {
    if (!fmt_ok(fmt) || cols < 0 || cols % block_elems_of(fmt)) return 0;
    return rowbytes(fmt, cols);
}

const char* lq_status_str(int s) {
    switch (s) {
        case LQ_OK: return "LQ_OK";
        case LQ_EINVAL: return "LQ_EINVAL: invalid argument";
        case LQ_EALIGN: return "LQ_EALIGN: misaligned pointer";
        case LQ_ESHAPE: return "LQ_ESHAPE: unsupported shape";
        case LQ_EWORKSPACE: return "LQ_EWORKSPACE: workspace too small";
        case LQ_ECUDA: return "LQ_ECUDA: CUDA error";
        case LQ_ETIMEOUT: return "LQ_ETIMEOUT: a bounded device wait ran out";
        case LQ_EUNSUPPORTED: return "LQ_EUNSUPPORTED: not implemented";
        default: return "unknown lq status";
    }
}

const char* lq_last_error(void) { return g_err; }

void lq_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

int lq_dequant(int fmt, const void* W, int64_t rows, int64_t cols, float* out, lq_stream_t stream) {
    g_err[0] = 0;
    int rc = check_mat(fmt, W, rows, cols, "W");
    if (rc) return rc;
    if (rows == 0) return LQ_OK;
    if ((rc = check_f32(out, "out"))) return rc;
    cudaError_t e = launch_dequant(fmt, static_cast<const uint8_t*>(W), rows, cols, out,
                                   reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "dequant launch");
}

static size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// The transform `pre` as its own launch: the rows written to pre.out.
static int prepass(const XPre& pre, const float* x, int batch, int64_t cols, cudaStream_t st) {
    cudaError_t e = pre.kind == GV_X_NORM ? launch_rmsnorm(x, pre.nw, pre.eps, pre.out, batch, cols, st)
                                          : launch_act_pairs(x, pre.out, (int64_t)batch * cols, pre.act, st);
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "x transform launch");
}

// run_segments with an optional transform of x: fused when the kernel that
// runs has it, else the transform first (into pre.out) and the segments
// reading that.
static int run_pre(std::vector<Seg>& segs, int B, int64_t cols, int batch, cudaStream_t st, const XPre* pre,
                   const float* x) {
    if (!pre) return run_segments(segs, B, cols, st);
    int rc = run_segments(segs, B, cols, st, pre);
    if (rc != NEEDS_PREPASS) return rc;
    if ((rc = prepass(*pre, x, batch, cols, st))) return rc;
    for (auto& s : segs) {
        s.x = pre->out;
        s.xact = ACT_NONE;
        s.xout = nullptr;
    }
    return run_segments(segs, B, cols, st);
}

// y = W.x, each output stored through seg_out (cap 0: as computed); x
// transformed first by pre (if given)
static int matvec_impl(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                       float cap, lq_stream_t stream, const XPre* pre = nullptr) {
    int rc = check_mat(fmt, W, rows, cols, "W");
    if (rc) return rc;
    if (batch < 1) return fail(LQ_EINVAL, "batch %d < 1", batch);
    if (rows == 0) return LQ_OK;
    if ((rc = check_f32(x, "x")) || (rc = check_f32(y, "y"))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (batch >= qmm_min_batch(fmt)) {
        std::vector<Seg> segs;
        for (int b0 = 0; b0 < batch; b0 += QMM_NT) {
            segs.push_back(plain_seg(fmt, W, rows, pre ? pre->out : x, y, rows, b0, std::min(QMM_NT, batch - b0)));
            segs.back().cap = cap;
        }
        if (qmm_eligible(segs, cols)) {
            if (pre && (rc = prepass(*pre, x, batch, cols, st))) return rc;
            return run_qmm(segs, cols, st);
        }
    }
    if (batch > 1 && batch <= GVW_MAX_X && !pre) {
        // all x rows in one pass of the column-chunked tensor-core kernel
        // (Q6_K), whatever width the CUDA-core kernel would take
        std::vector<Seg> one{plain_seg(fmt, W, rows, x, y, rows, 0, batch)};
        one.back().cap = cap;
        rc = run_gvw(one, cols, st, nullptr);
        if (rc != GV_NOT_ELIGIBLE) return rc;
    }
    const int B = batch_width(cols, batch, {fmt}, false);
    std::vector<Seg> segs;
    for (int b0 = 0; b0 < batch; b0 += B) {
        segs.push_back(plain_seg(fmt, W, rows, x, y, rows, b0, std::min(B, batch - b0)));
        segs.back().cap = cap;
    }
    return run_pre(segs, B, cols, batch, st, pre, x);
}

static int qkv_impl(int fq, const void* Wq, int64_t nq, int fk, const void* Wk, int64_t nk, int fv, const void* Wv,
                    int64_t nv, int64_t cols, const float* x, float* q, float* k, float* v, int batch,
                    lq_stream_t stream, const XPre* pre = nullptr) {
    int rc;
    if ((rc = check_mat(fq, Wq, nq, cols, "Wq")) || (rc = check_mat(fk, Wk, nk, cols, "Wk")) ||
        (rc = check_mat(fv, Wv, nv, cols, "Wv")))
        return rc;
    if (batch < 1) return fail(LQ_EINVAL, "batch %d < 1", batch);
    if (nq + nk + nv == 0) return LQ_OK;
    if ((rc = check_f32(x, "x"))) return rc;
    if ((nq && (rc = check_f32(q, "q"))) || (nk && (rc = check_f32(k, "k"))) ||
        (nv && (rc = check_f32(v, "v"))))
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (batch >= qmm_min_batch(fq)) {
        const float* xq = pre ? pre->out : x;
        std::vector<Seg> segs;
        for (int b0 = 0; b0 < batch; b0 += QMM_NT) {
            const int nb = std::min(QMM_NT, batch - b0);
            if (nq) segs.push_back(plain_seg(fq, Wq, nq, xq, q, nq, b0, nb));
            if (nk) segs.push_back(plain_seg(fk, Wk, nk, xq, k, nk, b0, nb));
            if (nv) segs.push_back(plain_seg(fv, Wv, nv, xq, v, nv, b0, nb));
        }
        if (qmm_eligible(segs, cols)) {
            if (pre && (rc = prepass(*pre, x, batch, cols, st))) return rc;
            return run_qmm(segs, cols, st);
        }
    }
    const int B = batch_width(cols, batch, {fq, fk, fv}, false);
    std::vector<Seg> segs;
    for (int b0 = 0; b0 < batch; b0 += B) {
        const int nb = std::min(B, batch - b0);
        if (nq) segs.push_back(plain_seg(fq, Wq, nq, x, q, nq, b0, nb));
        if (nk) segs.push_back(plain_seg(fk, Wk, nk, x, k, nk, b0, nb));
        if (nv) segs.push_back(plain_seg(fv, Wv, nv, x, v, nv, b0, nb));
    }
    return run_pre(segs, B, cols, batch, st, pre, x);
}

static int gate_up_impl(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* x, float* h, int batch,
                        int act, lq_stream_t stream, const XPre* pre = nullptr) {
    int rc = check_mat(fmt, Wgu, 2 * inter, cols, "Wgu");
    if (rc) return rc;
    if (batch < 1) return fail(LQ_EINVAL, "batch %d < 1", batch);
    if (act != LQ_ACT_GEGLU_TANH && act != LQ_ACT_SWIGLU) return fail(LQ_EINVAL, "act %d", act);
    if (inter == 0) return LQ_OK;
    if ((rc = check_f32(x, "x")) || (rc = check_f32(h, "h"))) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (batch >= qmm_min_batch(fmt)) {
        std::vector<Seg> segs;
        for (int b0 = 0; b0 < batch; b0 += QMM_NT) {
            Seg s = plain_seg(fmt, Wgu, inter, pre ? pre->out : x, h, inter, b0, std::min(QMM_NT, batch - b0));
            s.mode = MODE_PAIR_INTERLEAVED;
            s.act = act;
            segs.push_back(s);
        }
        if (qmm_eligible(segs, cols)) {
            if (pre && (rc = prepass(*pre, x, batch, cols, st))) return rc;
            return run_qmm(segs, cols, st);
        }
    }
    const int B = batch_width(cols, batch, {fmt}, true);
    std::vector<Seg> segs;
    for (int b0 = 0; b0 < batch; b0 += B) {
        Seg s = plain_seg(fmt, Wgu, inter, x, h, inter, b0, std::min(B, batch - b0));
        s.mode = MODE_PAIR_INTERLEAVED;
        s.act = act;
        segs.push_back(s);
    }
    return run_pre(segs, B, cols, batch, st, pre, x);
}

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

// Arguments of the fused input norm: weight, epsilon, the normalised rows'
// buffer (not overlapping x: the fused kernel stores it while others read x).
static int check_norm(const float* x, const float* nw, float eps, const float* xn, int batch, int64_t cols) {
    int rc;
    if ((rc = check_f32(nw, "norm_w")) || (rc = check_f32(xn, "xn"))) return rc;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(LQ_EINVAL, "eps %g", (double)eps);
    if (x && batch > 0 && cols > 0 && overlaps(x, (size_t)batch * cols * 4, xn, (size_t)batch * cols * 4))
        return fail(LQ_EINVAL, "xn overlaps x");
    return LQ_OK;
}

int lq_matvec(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y,
              int batch, lq_stream_t stream) {
    g_err[0] = 0;
    return matvec_impl(fmt, W, rows, cols, x, y, batch, 0.f, stream);
}

int lq_matvec_softcap(int fmt, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                      float cap, lq_stream_t stream) {
    g_err[0] = 0;
    if (!(cap > 0.f) || !std::isfinite(cap)) return fail(LQ_EINVAL, "soft-cap %g: not a finite positive value", (double)cap);
    return matvec_impl(fmt, W, rows, cols, x, y, batch, cap, stream);
}

int lq_matvec_act(int fmt, const void* W, int64_t rows, int64_t cols, const float* gu, float* h, float* y, int batch,
                  int act, lq_stream_t stream) {
    g_err[0] = 0;
    if (act != LQ_ACT_GEGLU_TANH && act != LQ_ACT_SWIGLU) return fail(LQ_EINVAL, "act %d", act);
    int rc;
    if ((rc = check_f32(h, "h"))) return rc;
    if (gu && batch > 0 && cols > 0 && overlaps(gu, (size_t)batch * cols * 8, h, (size_t)batch * cols * 4))
        return fail(LQ_EINVAL, "h overlaps gu");
    XPre pre;
    pre.kind = GV_X_ACT;
    pre.act = act;
    pre.out = h;
    return matvec_impl(fmt, W, rows, cols, gu, y, batch, 0.f, stream, &pre);
}

size_t lq_gemm_workspace_bytes(int64_t M, int64_t rows, int64_t cols) {
    if (M < 0 || rows < 0 || cols < 0) return 0;
    // the x image (hi and lo pieces, M padded to whole x tiles), s_n, 1 / t_r
    // and, when K is split, the partial sums
    const size_t mp = (size_t)((M + GEMM_TC_XN - 1) / GEMM_TC_XN) * GEMM_TC_XN;
    const int ks = gemm_tc_ksplit(rows, cols);
    return align256(mp * cols * 4) + align256(mp * 4) + align256((size_t)rows * 4) +
           (ks > 1 ? align256((size_t)ks * M * rows * 4) : 0);
}

// The tiled GEMM of lq_gemm and lq_gemm_gate_up_act: Y[n][r] (plain) or
// Y[n][i] = act(row 2i) * row 2i + 1 (pairs), W of `rows` rows.
static int gemm_tiled(int fmt, const void* W, int64_t rows, int64_t cols, const float* X, float* Y, int64_t ld_y,
                      int64_t M, int pairs, int act, void* workspace, size_t ws_bytes, lq_stream_t stream) {
    const size_t need = lq_gemm_workspace_bytes(M, rows, cols);
    if (!workspace || ws_bytes < need) return fail(LQ_EWORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    if (!al(workspace, 256)) return fail(LQ_EALIGN, "workspace not 256-byte aligned");
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    uint8_t* p = static_cast<uint8_t*>(workspace);
    GemmParams P;
    memset(&P, 0, sizeof P);
    P.W = static_cast<const uint8_t*>(W);
    P.rows = rows;
    P.cols = cols;
    P.rowbytes = rowbytes(fmt, cols);
    P.M = M;
    P.ld_y = ld_y;
    P.pairs = pairs;
    P.act = act;
    P.nmt = (int32_t)((M + GEMM_TC_XN - 1) / GEMM_TC_XN);
    if ((rc = tensor_map(&P.tmw, W, rows, P.rowbytes, P.rowbytes, (int)(P.rowbytes / (cols / 256) / 4), GEMM_TC_WR)))
        return rc;
    const size_t mp = (size_t)P.nmt * GEMM_TC_XN;
    P.ximg = p; p += align256(mp * cols * 4);
    P.sn = reinterpret_cast<float*>(p); p += align256(mp * 4);
    P.tinv = reinterpret_cast<float*>(p); p += align256((size_t)rows * 4);
    P.ksplit = gemm_tc_ksplit(rows, cols);
    P.part = P.ksplit > 1 ? reinterpret_cast<float*>(p) : nullptr;
    P.Y = Y;
    P.timeout_ns = g_timeout_ns.load();
    P.status = dev->status;
    cudaError_t e = gemm_tc_launch(fmt, P, X, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "gemm launch");
}

static bool gemm_is_tiled(int fmt, const void* W, int64_t cols, const float* X, int64_t M) {
    return (fmt == FMT_Q4_K || fmt == FMT_Q8_0) && cols % 256 == 0 && M >= LQ_GEMM_MIN_M && al(W, 16) && al(X, 16) &&
           rowbytes(fmt, cols) % 16 == 0;
}

int lq_gemm(int fmt, const void* W, int64_t rows, int64_t cols, const float* X, float* Y, int64_t M,
            void* workspace, size_t ws_bytes, lq_stream_t stream) {
    g_err[0] = 0;
    int rc = check_mat(fmt, W, rows, cols, "W");
    if (rc) return rc;
    if (M < 1 || M > (int64_t)1 << 24) return fail(LQ_EINVAL, "M %lld", (long long)M);
    if (rows == 0) return LQ_OK;
    if ((rc = check_f32(X, "X")) || (rc = check_f32(Y, "Y"))) return rc;
    if (!gemm_is_tiled(fmt, W, cols, X, M)) {
        // the batched matvec (a pass over the weights per 8 x rows)
        for (int64_t b0 = 0; b0 < M; b0 += 1 << 20) {
            const int nb = (int)std::min<int64_t>(1 << 20, M - b0);
            if ((rc = matvec_impl(fmt, W, rows, cols, X + b0 * cols, Y + b0 * rows, nb, 0.f, stream))) return rc;
        }
        return LQ_OK;
    }
    return gemm_tiled(fmt, W, rows, cols, X, Y, rows, M, 0, 0, workspace, ws_bytes, stream);
}

int lq_gemm_gate_up_act(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* X, float* H, int64_t M,
                        int act, void* workspace, size_t ws_bytes, lq_stream_t stream) {
    g_err[0] = 0;
    if (act != LQ_ACT_GEGLU_TANH && act != LQ_ACT_SWIGLU) return fail(LQ_EINVAL, "act %d", act);
    if (inter < 0 || inter > (int64_t)1 << 29) return fail(LQ_ESHAPE, "inter %lld", (long long)inter);
    int rc = check_mat(fmt, Wgu, 2 * inter, cols, "Wgu");
    if (rc) return rc;
    if (M < 1 || M > (int64_t)1 << 24) return fail(LQ_EINVAL, "M %lld", (long long)M);
    if (inter == 0) return LQ_OK;
    if ((rc = check_f32(X, "X")) || (rc = check_f32(H, "H"))) return rc;
    if (!gemm_is_tiled(fmt, Wgu, cols, X, M)) {
        // the batched gate+up kernels (a pass over the weights per 8 x rows)
        for (int64_t b0 = 0; b0 < M; b0 += 1 << 20) {
            const int nb = (int)std::min<int64_t>(1 << 20, M - b0);
            if ((rc = gate_up_impl(fmt, Wgu, inter, cols, X + b0 * cols, H + b0 * inter, nb, act, stream))) return rc;
        }
        return LQ_OK;
    }
    return gemm_tiled(fmt, Wgu, 2 * inter, cols, X, H, inter, M, 1, act, workspace, ws_bytes, stream);
}

static int gemv_dense(bool f16, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch,
                      lq_stream_t stream) {
    const int epc = f16 ? 8 : 4;
    if (rows < 0 || rows > (int64_t)1 << 30 || cols <= 0 || cols % epc)
        return fail(LQ_ESHAPE, "rows %lld cols %lld (cols a multiple of %d)", (long long)rows, (long long)cols, epc);
    if (batch < 1 || batch > 8) return fail(LQ_EINVAL, "batch %d (1..8)", batch);
    if ((int64_t)batch * cols * 4 > 200 * 1024) return fail(LQ_ESHAPE, "batch * cols too large for the x staging");
    if (rows == 0) return LQ_OK;
    if (!W) return fail(LQ_EINVAL, "W is null");
    int rc;
    if ((rc = check_f32(x, "x")) || (rc = check_f32(y, "y"))) return rc;
    if (!al(W, 16) || !al(x, 16)) return fail(LQ_EALIGN, "W and x must be 16-byte aligned");
    DevInfo* dev = nullptr;
    if ((rc = dev_info(&dev))) return rc;
    cudaError_t e = dense_gemv_launch(f16, W, rows, (int)cols, x, y, batch, dev->sms,
                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "dense gemv launch");
}

int lq_gemv_f16(const void* W, int64_t rows, int64_t cols, const float* x, float* y, int batch, lq_stream_t stream) {
    g_err[0] = 0;
    return gemv_dense(true, W, rows, cols, x, y, batch, stream);
}

int lq_gemv_f32(const float* W, int64_t rows, int64_t cols, const float* x, float* y, int batch, lq_stream_t stream) {
    g_err[0] = 0;
    return gemv_dense(false, W, rows, cols, x, y, batch, stream);
}

int lq_rmsnorm(const float* x, const float* w, float eps, float* out, int ntok, int64_t n, lq_stream_t stream) {
    g_err[0] = 0;
    if (ntok < 0 || n <= 0 || n > (int64_t)1 << 20) return fail(LQ_ESHAPE, "ntok %d n %lld", ntok, (long long)n);
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(LQ_EINVAL, "eps %g", (double)eps);
    int rc;
    if ((rc = check_f32(x, "x")) || (rc = check_f32(w, "w")) || (rc = check_f32(out, "out"))) return rc;
    if (ntok == 0) return LQ_OK;
    cudaError_t e = launch_rmsnorm(x, w, eps, out, ntok, n, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "rmsnorm launch");
}

int lq_qkv_mixed(int fq, const void* Wq, int64_t nq, int fk, const void* Wk, int64_t nk, int fv,
                 const void* Wv, int64_t nv, int64_t cols, const float* x, float* q, float* k,
                 float* v, int batch, lq_stream_t stream) {
    g_err[0] = 0;
    return qkv_impl(fq, Wq, nq, fk, Wk, nk, fv, Wv, nv, cols, x, q, k, v, batch, stream);
}

int lq_qkv_mixed_rmsnorm(int fq, const void* Wq, int64_t nq, int fk, const void* Wk, int64_t nk, int fv,
                         const void* Wv, int64_t nv, int64_t cols, const float* x, const float* norm_w, float eps,
                         float* xn, float* q, float* k, float* v, int batch, lq_stream_t stream) {
    g_err[0] = 0;
    int rc = check_norm(x, norm_w, eps, xn, batch, cols);
    if (rc) return rc;
    XPre pre;
    pre.kind = GV_X_NORM;
    pre.nw = norm_w;
    pre.eps = eps;
    pre.out = xn;
    return qkv_impl(fq, Wq, nq, fk, Wk, nk, fv, Wv, nv, cols, x, q, k, v, batch, stream, &pre);
}

int lq_pack_gate_up(int fmt, const void* Wg, const void* Wu, int64_t inter, int64_t cols,
                    void* Wgu_out, lq_stream_t stream) {
    g_err[0] = 0;
    int rc;
    if ((rc = check_mat(fmt, Wg, inter, cols, "Wg")) || (rc = check_mat(fmt, Wu, inter, cols, "Wu")))
        return rc;
    if (inter == 0) return LQ_OK;
    if (!Wgu_out) return fail(LQ_EINVAL, "Wgu_out is null");
    if (!al(Wgu_out, 2)) return fail(LQ_EALIGN, "Wgu_out not 2-byte aligned");
    cudaError_t e = launch_interleave(static_cast<const uint8_t*>(Wg), static_cast<const uint8_t*>(Wu),
                                      inter, rowbytes(fmt, cols), static_cast<uint8_t*>(Wgu_out),
                                      reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "interleave launch");
}

int lq_ffn_gate_up_act(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* x,
                       float* h, int batch, int act, lq_stream_t stream) {
    g_err[0] = 0;
    return gate_up_impl(fmt, Wgu, inter, cols, x, h, batch, act, stream);
}

int lq_ffn_gate_up_act_rmsnorm(int fmt, const void* Wgu, int64_t inter, int64_t cols, const float* x,
                               const float* norm_w, float eps, float* xn, float* h, int batch, int act,
                               lq_stream_t stream) {
    g_err[0] = 0;
    int rc = check_norm(x, norm_w, eps, xn, batch, cols);
    if (rc) return rc;
    XPre pre;
    pre.kind = GV_X_NORM;
    pre.nw = norm_w;
    pre.eps = eps;
    pre.out = xn;
    return gate_up_impl(fmt, Wgu, inter, cols, x, h, batch, act, stream, &pre);
}

int lq_ffn(int fmt_gu, const void* Wgu, int fmt_down, const void* Wd, int64_t inter, int64_t hidden,
           const float* x, float* h, float* y, int batch, int act, lq_stream_t stream) {
    g_err[0] = 0;
    int rc;
    if ((rc = check_mat(fmt_gu, Wgu, 2 * inter, hidden, "Wgu")) ||
        (rc = check_mat(fmt_down, Wd, hidden, inter, "Wd")))
        return rc;
    if (inter == 0 || hidden == 0) return fail(LQ_ESHAPE, "inter %lld hidden %lld", (long long)inter, (long long)hidden);
    if (batch < 1) return fail(LQ_EINVAL, "batch %d < 1", batch);
    if (act != LQ_ACT_GEGLU_TANH && act != LQ_ACT_SWIGLU) return fail(LQ_EINVAL, "act %d", act);
    if ((rc = check_f32(x, "x")) || (rc = check_f32(h, "h")) || (rc = check_f32(y, "y"))) return rc;
    if ((rc = lq_ffn_gate_up_act(fmt_gu, Wgu, inter, hidden, x, h, batch, act, stream))) return rc;
    return lq_matvec(fmt_down, Wd, hidden, inter, h, y, batch, stream);
}

size_t lq_moe_ffn_ex_workspace_bytes(int E, int topk, int ntok, int64_t hidden, int64_t inter, int n_shared,
                                     int64_t inter_s) {
    if (E < 1 || topk < 1 || ntok < 0 || hidden < 0 || inter < 0 || n_shared < 0 || inter_s < 0) return 0;
    const size_t ns = (size_t)ntok * topk;
    size_t b = align256(ns * 4) * 4 + align256((size_t)E * 4) * 2 + align256(ns * inter * 4) +
               align256(ns * hidden * 4);
    if (n_shared > 0)
        b += align256((size_t)ntok * 4) + align256((size_t)n_shared * ntok * inter_s * 4) +
             align256((size_t)n_shared * ntok * hidden * 4);
    return b;
}

size_t lq_moe_workspace_bytes(int E, int topk, int ntok, int64_t hidden, int64_t inter) {
    return lq_moe_ffn_ex_workspace_bytes(E, topk, ntok, hidden, inter, 0, 0);
}

int lq_moe_ffn_ex(const float* router, int E, int topk, int norm_topk_prob, int fmt, const void* const* W1,
                  const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter, int n_shared,
                  const void* const* Ws1, const void* const* Ws3, const void* const* Ws2, int64_t inter_s,
                  const float* shared_gate, const float* X, float* Y, int ntok, int32_t* topk_idx, float* topk_w,
                  void* workspace, size_t ws_bytes, lq_stream_t stream) {
    g_err[0] = 0;
    int rc = moe_validate(router, E, topk, norm_topk_prob, fmt, W1, W3, W2, hidden, inter, n_shared, Ws1, Ws3,
                          Ws2, inter_s, shared_gate, X, Y, ntok, topk_idx, topk_w);
    if (rc || ntok == 0) return rc;
    const size_t need = lq_moe_ffn_ex_workspace_bytes(E, topk, ntok, hidden, inter, n_shared, inter_s);
    if (!workspace || ws_bytes < need)
        return fail(LQ_EWORKSPACE, "workspace %zu < %zu bytes", ws_bytes, need);
    if (!al(workspace, 256)) return fail(LQ_EALIGN, "workspace not 256-byte aligned");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    const size_t ns = (size_t)ntok * topk;
    uint8_t* p = static_cast<uint8_t*>(workspace);
    MoeWs ws;
    memset(&ws, 0, sizeof ws);
    ws.idx = reinterpret_cast<int32_t*>(p); p += align256(ns * 4);
    ws.w = reinterpret_cast<float*>(p); p += align256(ns * 4);
    ws.tok_of = reinterpret_cast<int32_t*>(p); p += align256(ns * 4);
    ws.slot_row = reinterpret_cast<int32_t*>(p); p += align256(ns * 4);
    ws.grp_off = reinterpret_cast<int32_t*>(p); p += align256((size_t)E * 4);
    ws.grp_cnt = reinterpret_cast<int32_t*>(p); p += align256((size_t)E * 4);
    ws.hbuf = reinterpret_cast<float*>(p); p += align256(ns * inter * 4);
    ws.ybuf = reinterpret_cast<float*>(p); p += align256(ns * hidden * 4);
    if (n_shared > 0) {
        ws.sgate = reinterpret_cast<float*>(p); p += align256((size_t)ntok * 4);
        ws.hsh = reinterpret_cast<float*>(p); p += align256((size_t)n_shared * ntok * inter_s * 4);
        ws.ysh = reinterpret_cast<float*>(p);
        if (!shared_gate) ws.sgate = nullptr;
    }
    ws.nshared = n_shared;
    ws.norm = norm_topk_prob;
    if (topk_idx) ws.idx = topk_idx;
    if (topk_w) ws.w = topk_w;

    cudaError_t e = launch_moe_route(router, E, hidden, X, ntok, topk, shared_gate, ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "moe route launch");

    // Routed experts: one segment per (expert, chunk of B grouped rows), the
    // row count read from the routing on the device.  Shared experts: dense
    // segments over all tokens (chunks of B), in the same launch when they
    // take the same kernel and (for down) the same width.
    const bool tc = moe_tc_ok(fmt, ntok, hidden, inter, W1, W3, W2, E, X);
    const bool tcs = n_shared > 0 && moe_tc_ok(fmt, ntok, hidden, inter_s, Ws1, Ws3, Ws2, n_shared, X);
    auto shared_seg = [&](int ex, bool up, int b0, int nb) {
        Seg s;
        memset(&s, 0, sizeof s);
        if (up) {
            s.w = static_cast<const uint8_t*>(Ws1[ex]);
            s.w2 = static_cast<const uint8_t*>(Ws3[ex]);
            s.x = X;
            s.y = ws.hsh + (int64_t)ex * ntok * inter_s;
            s.ld_y = inter_s;
            s.nout = (int32_t)inter_s;
            s.mode = MODE_PAIR_TWO;
            s.act = ACT_SWIGLU;
        } else {
            s.w = static_cast<const uint8_t*>(Ws2[ex]);
            s.x = ws.hsh + (int64_t)ex * ntok * inter_s;
            s.y = ws.ysh + (int64_t)ex * ntok * hidden;
            s.ld_y = hidden;
            s.nout = (int32_t)hidden;
            s.mode = MODE_PLAIN;
        }
        s.fmt = fmt;
        s.b0 = b0;
        s.nbatch = nb;
        return s;
    };
    auto run = [&](std::vector<Seg>& segs, bool t, int B, int64_t cols) {
        if (segs.empty()) return (int)LQ_OK;
        return t ? run_qmm(segs, cols, st) : run_segments(segs, B, cols, st);
    };
    // grouped expert gate+up (+SwiGLU)
    {
        const int B = tc ? QMM_NT : batch_width(hidden, ntok, {fmt}, true);
        const int Bs = tcs ? QMM_NT : batch_width(hidden, ntok, {fmt}, true);
        std::vector<Seg> segs, ssegs;
        for (int c = 0; c * B < ntok; ++c)
            for (int ex = 0; ex < E; ++ex) {
                Seg s;
                memset(&s, 0, sizeof s);
                s.w = static_cast<const uint8_t*>(W1[ex]);
                s.w2 = static_cast<const uint8_t*>(W3[ex]);
                s.x = X;
                s.xmap = ws.tok_of;
                s.y = ws.hbuf;
                s.boff = ws.grp_off + ex;
                s.bcnt = ws.grp_cnt + ex;
                s.ld_y = inter;
                s.nout = (int32_t)inter;
                s.fmt = fmt;
                s.mode = MODE_PAIR_TWO;
                s.act = ACT_SWIGLU;
                s.b0 = c * B;
                segs.push_back(s);
            }
        std::vector<Seg>& dst = (tcs == tc && Bs == B) ? segs : ssegs;
        for (int c = 0; c * Bs < ntok; ++c)
            for (int ex = 0; ex < n_shared; ++ex) dst.push_back(shared_seg(ex, true, c * Bs, std::min(Bs, ntok - c * Bs)));
        if ((rc = run(segs, tc, B, hidden)) || (rc = run(ssegs, tcs, Bs, hidden))) return rc;
    }
    // grouped expert down: x rows are the grouped hidden activations
    {
        const int B = tc ? QMM_NT : batch_width(inter, ntok, {fmt}, false);
        const int Bs = tcs ? QMM_NT : batch_width(inter_s, ntok, {fmt}, false);
        std::vector<Seg> segs, ssegs;
        for (int c = 0; c * B < ntok; ++c)
            for (int ex = 0; ex < E; ++ex) {
                Seg s;
                memset(&s, 0, sizeof s);
                s.w = static_cast<const uint8_t*>(W2[ex]);
                s.x = ws.hbuf;
                s.y = ws.ybuf;
                s.boff = ws.grp_off + ex;
                s.bcnt = ws.grp_cnt + ex;
                s.ld_y = hidden;
                s.nout = (int32_t)hidden;
                s.fmt = fmt;
                s.mode = MODE_PLAIN;
                s.b0 = c * B;
                segs.push_back(s);
            }
        std::vector<Seg>& dst = (tcs == tc && Bs == B && inter_s == inter) ? segs : ssegs;
        for (int c = 0; c * Bs < ntok; ++c)
            for (int ex = 0; ex < n_shared; ++ex) dst.push_back(shared_seg(ex, false, c * Bs, std::min(Bs, ntok - c * Bs)));
        if ((rc = run(segs, tc, B, inter)) || (rc = run(ssegs, tcs, Bs, inter_s))) return rc;
    }
    e = launch_moe_combine(ws.ybuf, hidden, ntok, topk, ws, Y, st);
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "moe combine launch");
}

int lq_moe_ffn(const float* router, int E, int topk, int fmt, const void* const* W1,
               const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter,
               const float* X, float* Y, int ntok, int32_t* topk_idx, float* topk_w,
               void* workspace, size_t ws_bytes, lq_stream_t stream) {
    return lq_moe_ffn_ex(router, E, topk, 1, fmt, W1, W3, W2, hidden, inter, 0, nullptr, nullptr, nullptr, 0,
                         nullptr, X, Y, ntok, topk_idx, topk_w, workspace, ws_bytes, stream);
}

// No-allocation variant: the scratch is a static device array of this
// module, its address looked up per device and context (with that device
// current), again after a context change such as cudaDeviceReset.
int lq_moe_ffn_static(const float* router, int E, int topk, int fmt, const void* const* W1,
                      const void* const* W3, const void* const* W2, int64_t hidden, int64_t inter,
                      const float* X, float* Y, int ntok, int32_t* topk_idx, float* topk_w,
                      lq_stream_t stream) {
    g_err[0] = 0;
    int rc = moe_validate(router, E, topk, 1, fmt, W1, W3, W2, hidden, inter, 0, nullptr, nullptr, nullptr, 0,
                          nullptr, X, Y, ntok, topk_idx, topk_w);
    if (rc) return rc;
    const size_t need = lq_moe_workspace_bytes(E, topk, ntok, hidden, inter);
    if (need > (size_t)LQ_MOE_STATIC_SCRATCH_BYTES)
        return fail(LQ_EWORKSPACE, "MoE needs %zu bytes of scratch; the static scratch holds %zu", need,
                    (size_t)LQ_MOE_STATIC_SCRATCH_BYTES);
    if (ntok == 0) return LQ_OK;
    int d = 0;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (d < 0 || d >= kMaxDevices) return fail(LQ_EINVAL, "device %d out of range", d);
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_moe_scratch_mu);
        const unsigned long long ctx = current_ctx_id();
        if (!g_moe_scratch_ptr[d] || ctx == 0 || ctx != g_moe_scratch_ctx[d]) {
            void* ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_moe_scratch);
            if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static MoE scratch)");
            g_moe_scratch_ptr[d] = ptr;
            g_moe_scratch_ctx[d] = current_ctx_id();
        }
        scratch = g_moe_scratch_ptr[d];
    }
    return lq_moe_ffn(router, E, topk, fmt, W1, W3, W2, hidden, inter, X, Y, ntok, topk_idx, topk_w,
                      scratch, (size_t)LQ_MOE_STATIC_SCRATCH_BYTES, stream);
}

int lq_device_status(lq_stream_t stream, uint32_t* bits) {
    g_err[0] = 0;
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    (void)stream;
    cudaError_t e = cudaDeviceSynchronize();     // the word is shared by every stream's launches
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    unsigned v = 0;
    e = cudaMemcpy(&v, dev->status, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read status");
    const unsigned zero = 0;
    e = cudaMemcpy(dev->status, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear status");
    if (bits) *bits = v;
    return (v & STATUS_TIMEOUT) ? fail(LQ_ETIMEOUT, "device status 0x%x", v) : LQ_OK;
}

int lq_probe_timeout(uint64_t timeout_ns, lq_stream_t stream) {
    g_err[0] = 0;
    DevInfo* dev = nullptr;
    int rc = dev_info(&dev);
    if (rc) return rc;
    cudaError_t e = launch_timeout_probe(timeout_ns, dev->status, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? LQ_OK : cuda_fail(e, "probe launch");
}

}  // extern "C"
