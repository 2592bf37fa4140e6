// api.cu - the C ABI of include/locks.h: argument validation, workspace
// layout and kernel launches. No allocation, no host synchronisation (except
// locks_get_device_status), so every compute call can be captured in a CUDA
// graph.
#include <algorithm>
#include <atomic>
#include <mutex>

#include "locks_internal.h"

namespace {

constexpr size_t kAlign = 256;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;   // 2 s
constexpr int kMaxDevices = 64;

std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

int num_sms(int dev) {
    static std::atomic<int> cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = cache[dev].load();
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(v);
    return v;
}

// Cluster size for the select/attend kernels: 16 or 8 (two CTAs of either share an SM when
// their shared memory allows, and the hardware then packs them so), or 12 (one CTA per
// SM). A cluster of CL CTAs handles one (sequence, kv head) segment; when the segments do
// not all fit at once the launch runs in waves, so the choice minimises
// waves x (pages per SM + a fixed per-CTA cost in page units), for the selection launch's
// shared memory. Attention-only launches that do not split take the same size, so that
// they divide a selection among CTAs and warps as the fused launch does. Residency counts
// come from the occupancy API, cached per (device, mode, group bound, pages).
// locks_set_select_cluster pins the size.
std::atomic<int> g_select_cluster{0};
constexpr int kClusterSizes[3] = {16, 12, 8};

struct ClusterFit {
    int active[3];    // co-resident clusters, per kClusterSizes entry (0: cannot launch)
    int per_sm[3];    // CTAs of the launch sharing an SM
};

ClusterFit cluster_fit(int dev, const locks_dims_t* d, locks::SAMode mode) {
    struct Entry {
        int dev, mode, gbound, max_pages;
        ClusterFit fit;
    };
    static std::mutex mu;
    static Entry table[128];
    static int n = 0;
    const int g = d->num_q_heads / d->num_kv_heads;
    const int gbound = g <= 4 ? 4 : 16;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (table[i].dev == dev && table[i].mode == static_cast<int>(mode) && table[i].gbound == gbound &&
            table[i].max_pages == d->max_pages_per_seq)
            return table[i].fit;
    ClusterFit f;
    for (int i = 0; i < 3; ++i) {
        const int cl = kClusterSizes[i];
        f.active[i] = locks::select_attend_active_clusters(d->max_pages_per_seq, mode, g, cl);
        f.per_sm[i] = locks::select_attend_ctas_per_sm(d->max_pages_per_seq, mode, cl);
    }
    if (n < 128) table[n++] = {dev, static_cast<int>(mode), gbound, d->max_pages_per_seq, f};
    return f;
}

int cluster_size(int dev, const locks_dims_t* d) {
    const int pinned = g_select_cluster.load();
    if (pinned != 0) return pinned;
    const ClusterFit f = cluster_fit(dev, d, locks::SAMode::kSelectAttend);
    const long segs = static_cast<long>(d->batch) * d->num_kv_heads;
    int best = 16;
    double best_cost = 1e300;
    for (int i = 0; i < 3; ++i) {
        if (f.active[i] <= 0) continue;
        const int cl = kClusterSizes[i];
        const long waves = (segs + f.active[i] - 1) / f.active[i];
        const double cost = static_cast<double>(waves) *
                            (static_cast<double>(f.per_sm[i]) * ((d->max_pages_per_seq + cl - 1) / cl) + 2048.0);
        if (cost < best_cost) {
            best_cost = cost;
            best = cl;
        }
    }
    return best;
}

locks::DeviceStatus status_of(void* ws) {
    locks::DeviceStatus st;
    st.word = reinterpret_cast<int32_t*>(ws);
    st.wait_limit_ns = g_wait_limit_ns.load();
    return st;
}

int validate_dims(const locks_dims_t* d) {
    if (!d) return LOCKS_ERR_INVALID_ARG;
    if (d->head_dim != LOCKS_HEAD_DIM || d->page_size != LOCKS_PAGE_SIZE || d->rank != LOCKS_RANK)
        return LOCKS_ERR_UNSUPPORTED;
    if (d->batch < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->max_pages_per_seq < 0 ||
        d->num_phys_pages < 0)
        return LOCKS_ERR_INVALID_ARG;
    if (d->num_q_heads % d->num_kv_heads != 0) return LOCKS_ERR_INVALID_ARG;
    const int hkv = d->num_kv_heads;
    if (hkv != 1 && hkv != 2 && hkv != 4 && hkv != 8) return LOCKS_ERR_UNSUPPORTED;
    if (d->num_q_heads / hkv > LOCKS_MAX_GROUP) return LOCKS_ERR_UNSUPPORTED;
    if (d->batch > 0 && d->max_pages_per_seq > 0 && d->num_phys_pages <= 0) return LOCKS_ERR_INVALID_ARG;
    return LOCKS_OK;
}

// Bytes of the scorer's LSE partials: one (max, sum exp) pair per (sequence, query head,
// scorer CTA, consumer-warp slot), for the largest scorer grid.
size_t partials_bytes(const locks_dims_t* d) {
    const int g = d->num_q_heads / d->num_kv_heads;
    return static_cast<size_t>(d->batch) * d->num_q_heads * locks::kMaxScorerCtas *
           locks::slot_warps(d->num_kv_heads, g) * 8;
}

// Grid of the scorer launch for these dims on a device with `sms` SMs available to it.
int scorer_grid(const locks_dims_t* d, int sms) {
    const int np = locks::kStageUnits / d->num_kv_heads;
    const int nchunks = (d->max_pages_per_seq + np - 1) / np;
    return locks::score_grid(d->batch * nchunks, sms);
}

int k_cap_of(const locks_dims_t* d, int32_t budget) {
    int k = budget / LOCKS_PAGE_SIZE;
    if (k > d->max_pages_per_seq) k = d->max_pages_per_seq;
    return k < 1 ? 1 : k;
}

struct WsLayout {
    size_t status, scores, partials, selected, n_selected, split_cnt, split_part, split_end, total;
};
WsLayout ws_layout(const locks_dims_t* d, int32_t budget) {
    WsLayout w;
    const size_t B = static_cast<size_t>(d->batch);
    w.status = 0;
    w.scores = kAlign;
    w.partials = w.scores + align_up(B * d->num_q_heads * static_cast<size_t>(d->max_pages_per_seq) * 4);
    w.selected = w.partials + align_up(partials_bytes(d));
    w.n_selected = w.selected + align_up(B * d->num_kv_heads * static_cast<size_t>(k_cap_of(d, budget)) * 4);
    w.total = w.n_selected + align_up(B * d->num_kv_heads * 4);
    // split attention (attention-only calls, never alongside the regions above)
    w.split_cnt = kAlign;
    w.split_part = w.split_cnt + align_up(B * d->num_q_heads * 4);
    w.split_end =
        w.split_part + align_up(B * d->num_q_heads * locks::kMaxSplits * locks::kSplitPartFloats * sizeof(float));
    if (w.split_end > w.total) w.total = w.split_end;
    return w;
}

// An attention-only launch over up to k_cap pages per segment: the cluster size and
// the number of clusters per segment. Long selections are split over more clusters
// (merged through the workspace) while all of them stay co-resident and each CTA
// keeps at least kMinSplitPages pages; otherwise one cluster per segment.
constexpr int kMinSplitPages = 64;
void attention_plan(int dev, const locks_dims_t* d, int k_cap, bool can_split, int* cl, int* splits) {
    *cl = cluster_size(dev, d);
    *splits = 1;
    if (!can_split) return;
    const ClusterFit f = cluster_fit(dev, d, locks::SAMode::kAttend);
    const long segs = static_cast<long>(d->batch) * d->num_kv_heads;
    long best = *cl;
    for (int c : {16, 8}) {
        const long act = c == 16 ? f.active[0] : f.active[2];
        long sp = std::min<long>(locks::kMaxSplits, act / std::max<long>(segs, 1));
        sp = std::min<long>(sp, k_cap / (static_cast<long>(c) * kMinSplitPages));
        if (sp >= 2 && c * sp > best) {
            best = c * sp;
            *cl = c;
            *splits = static_cast<int>(sp);
        }
    }
}

int check_ws(void* ws, size_t bytes, size_t need) {
    if (!ws) return need == 0 ? LOCKS_OK : LOCKS_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(ws, kAlign)) return LOCKS_ERR_INVALID_ARG;
    if (bytes < need) return LOCKS_ERR_WORKSPACE_TOO_SMALL;
    return LOCKS_OK;
}

int check_summaries(const locks_summaries_t& s) {
    if (!s.mu || !s.basis || !s.coef || !s.scales) return LOCKS_ERR_INVALID_ARG;
    if (!aligned(s.mu, 16) || !aligned(s.basis, 16) || !aligned(s.coef, 16) || !aligned(s.scales, 8))
        return LOCKS_ERR_INVALID_ARG;
    return LOCKS_OK;
}

int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return LOCKS_OK;
    cudaGetLastError();
    return LOCKS_ERR_CUDA;
}

bool select_fits(int max_pages, locks::SAMode mode) {
    return locks::select_attend_smem_bytes(max_pages, 8, mode) <= 200 * 1024;
}

// reserve_sms: SMs the persistent scorer leaves free (for concurrent one-page builds).
int score_impl(const locks_dims_t* dims, const float* q, locks_summaries_t s, const int32_t* page_table,
               const int32_t* seq_pages, float* scores, float* partials, void* ws, cudaStream_t stream,
               int reserve_sms = 0) {
    const int dev = current_device();
    if (dev < 0) return LOCKS_ERR_CUDA;
    locks::ScoreArgs a;
    a.q = q;
    a.mu = s.mu;
    a.basis = s.basis;
    a.coef = s.coef;
    a.scales = s.scales;
    a.page_table = page_table;
    a.seq_pages = seq_pages;
    a.scores = scores;
    a.lse_partials = partials;
    a.batch = dims->batch;
    a.hq = dims->num_q_heads;
    a.hkv = dims->num_kv_heads;
    a.max_pages = dims->max_pages_per_seq;
    a.num_phys = dims->num_phys_pages;
    a.st = status_of(ws);
    return cuda_status(locks::launch_score(a, std::max(1, num_sms(dev) - reserve_sms), stream));
}

locks::SelectAttendArgs sa_args(const locks_dims_t* dims, void* ws) {
    locks::SelectAttendArgs a = {};
    a.batch = dims->batch;
    a.hq = dims->num_q_heads;
    a.hkv = dims->num_kv_heads;
    a.max_pages = dims->max_pages_per_seq;
    a.num_phys = dims->num_phys_pages;
    a.st = status_of(ws);
    return a;
}

int select_attend_impl(const locks_dims_t* dims, const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                       const int32_t* page_table, const float* scores, const float* partials,
                       const int32_t* seq_pages, const int32_t* tail_tokens,
                       int32_t budget_tokens, int32_t* selected, int32_t* n_selected, uint16_t* out, float* lse,
                       void* workspace, cudaStream_t st, int reserve_sms = 0) {
    const int dev = current_device();
    if (dev < 0) return LOCKS_ERR_CUDA;
    locks::SelectAttendArgs a = sa_args(dims, workspace);
    a.scores = scores;
    a.lse_partials = partials;
    a.score_grid = scorer_grid(dims, std::max(1, num_sms(dev) - reserve_sms));
    a.seq_pages = seq_pages;
    a.selected = selected;
    a.n_selected = n_selected;
    a.sel_keys = nullptr;
    a.budget_pages = budget_tokens / LOCKS_PAGE_SIZE;
    a.k_cap = k_cap_of(dims, budget_tokens);
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.page_table = page_table;
    a.tail_tokens = tail_tokens;
    a.out = out;
    a.lse = lse;
    const int cl = cluster_size(dev, dims);
    return cuda_status(locks::launch_select_attend(a, locks::SAMode::kSelectAttend, cl, st));
}

}  // namespace

extern "C" {

int locks_version(void) { return 10000; }

const char* locks_status_string(int status) {
    switch (status) {
        case LOCKS_OK: return "ok";
        case LOCKS_ERR_INVALID_ARG: return "invalid argument";
        case LOCKS_ERR_UNSUPPORTED: return "unsupported size";
        case LOCKS_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case LOCKS_ERR_CUDA: return "CUDA launch or runtime error";
        case LOCKS_ERR_TIMEOUT: return "device wait timed out";
        case LOCKS_ERR_BAD_INDEX: return "page index out of range on the device";
        default: return "unknown status";
    }
}

int locks_k_cap(const locks_dims_t* dims, int32_t budget_tokens, int32_t* k_cap) {
    if (!dims || !k_cap || budget_tokens < 0) return LOCKS_ERR_INVALID_ARG;
    *k_cap = k_cap_of(dims, budget_tokens);
    return LOCKS_OK;
}

int locks_workspace_size(const locks_dims_t* dims, int32_t budget_tokens, size_t* bytes) {
    if (!bytes || budget_tokens < 0) return LOCKS_ERR_INVALID_ARG;
    const int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    *bytes = ws_layout(dims, budget_tokens).total;
    return LOCKS_OK;
}

int locks_lse_partials_size(const locks_dims_t* dims, size_t* bytes) {
    if (!bytes) return LOCKS_ERR_INVALID_ARG;
    const int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    *bytes = partials_bytes(dims);
    return LOCKS_OK;
}

int locks_set_wait_limit_ns(uint64_t ns) {
    g_wait_limit_ns.store(ns == 0 ? kDefaultWaitNs : ns);
    return LOCKS_OK;
}

int locks_set_select_cluster(int32_t cluster) {
    if (cluster != 0 && cluster != 8 && cluster != 12 && cluster != 16) return LOCKS_ERR_INVALID_ARG;
    g_select_cluster.store(cluster);
    return LOCKS_OK;
}

int locks_build_summaries(const locks_dims_t* dims, const uint16_t* k_cache, const int32_t* phys_page_ids,
                          int32_t n_pages, locks_summaries_t summaries, void* workspace, size_t workspace_bytes,
                          void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (n_pages < 0) return LOCKS_ERR_INVALID_ARG;
    if (n_pages == 0) return LOCKS_OK;
    if (!k_cache || !phys_page_ids || !aligned(k_cache, 16)) return LOCKS_ERR_INVALID_ARG;
    if ((v = check_summaries(summaries)) != LOCKS_OK) return v;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    const int dev = current_device();
    if (dev < 0) return LOCKS_ERR_CUDA;
    locks::BuildArgs a;
    a.k_cache = k_cache;
    a.phys_page_ids = phys_page_ids;
    a.n_pages = n_pages;
    a.hkv = dims->num_kv_heads;
    a.num_phys = dims->num_phys_pages;
    a.mu = summaries.mu;
    a.basis = summaries.basis;
    a.coef = summaries.coef;
    a.scales = summaries.scales;
    a.st = status_of(workspace);
    return cuda_status(locks::launch_build(a, num_sms(dev), static_cast<cudaStream_t>(stream)));
}

int locks_score_pages(const locks_dims_t* dims, const float* q, locks_summaries_t summaries,
                      const int32_t* page_table, const int32_t* seq_pages, float* scores, float* lse_partials,
                      void* workspace, size_t workspace_bytes, void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (dims->batch == 0 || dims->max_pages_per_seq == 0) return LOCKS_OK;
    if (!q || !page_table || !seq_pages || !scores || !aligned(q, 16)) return LOCKS_ERR_INVALID_ARG;
    if (lse_partials && !aligned(lse_partials, 16)) return LOCKS_ERR_INVALID_ARG;
    if ((v = check_summaries(summaries)) != LOCKS_OK) return v;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    return score_impl(dims, q, summaries, page_table, seq_pages, scores, lse_partials, workspace,
                      static_cast<cudaStream_t>(stream));
}

int locks_select_pages(const locks_dims_t* dims, const float* scores, const float* lse_partials,
                       const int32_t* seq_pages, int32_t budget_tokens, int32_t* selected, int32_t* n_selected,
                       float* sel_keys, void* workspace, size_t workspace_bytes, void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (budget_tokens < 0) return LOCKS_ERR_INVALID_ARG;
    if (dims->batch == 0) return LOCKS_OK;
    if (!scores || !seq_pages || !selected || !n_selected) return LOCKS_ERR_INVALID_ARG;
    if (lse_partials && !aligned(lse_partials, 16)) return LOCKS_ERR_INVALID_ARG;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    if (!select_fits(dims->max_pages_per_seq, locks::SAMode::kSelect)) return LOCKS_ERR_UNSUPPORTED;
    const int dev = current_device();
    if (dev < 0) return LOCKS_ERR_CUDA;
    locks::SelectAttendArgs a = sa_args(dims, workspace);
    a.scores = scores;
    a.lse_partials = lse_partials;
    a.score_grid = scorer_grid(dims, num_sms(dev));
    a.seq_pages = seq_pages;
    a.selected = selected;
    a.n_selected = n_selected;
    a.sel_keys = sel_keys;
    a.budget_pages = budget_tokens / LOCKS_PAGE_SIZE;
    a.k_cap = k_cap_of(dims, budget_tokens);
    const int cl = cluster_size(dev, dims);
    return cuda_status(locks::launch_select_attend(a, locks::SAMode::kSelect, cl, static_cast<cudaStream_t>(stream)));
}

int locks_sparse_attention(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, const int32_t* page_table, const int32_t* selected,
                           const int32_t* n_selected, int32_t k_cap, uint16_t* out, float* lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (k_cap < 1) return LOCKS_ERR_INVALID_ARG;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !k_cache || !v_cache || !page_table || !selected || !n_selected || !out) return LOCKS_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return LOCKS_ERR_INVALID_ARG;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    const int dev = current_device();
    if (dev < 0) return LOCKS_ERR_CUDA;
    locks::SelectAttendArgs a = sa_args(dims, workspace);
    a.selected = const_cast<int32_t*>(selected);
    a.n_selected = const_cast<int32_t*>(n_selected);
    a.k_cap = k_cap;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.page_table = page_table;
    a.out = out;
    a.lse = lse;
    const WsLayout L = ws_layout(dims, k_cap * LOCKS_PAGE_SIZE);
    const bool can_split = workspace && workspace_bytes >= L.split_end;
    int cl = 16, splits = 1;
    attention_plan(dev, dims, k_cap, can_split, &cl, &splits);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (splits > 1) {
        uint8_t* base = static_cast<uint8_t*>(workspace);
        a.splits = splits;
        a.attn_cnt = reinterpret_cast<int32_t*>(base + L.split_cnt);
        a.attn_part = reinterpret_cast<float*>(base + L.split_part);
        v = cuda_status(cudaMemsetAsync(a.attn_cnt, 0, static_cast<size_t>(dims->batch) * dims->num_q_heads * 4, st));
        if (v != LOCKS_OK) return v;
    }
    return cuda_status(locks::launch_select_attend(a, locks::SAMode::kAttend, cl, st));
}

int locks_select_attend(const locks_dims_t* dims, const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* page_table, const float* scores, const float* lse_partials,
                        const int32_t* seq_pages, int32_t budget_tokens, int32_t* selected, int32_t* n_selected,
                        uint16_t* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    return locks_select_attend_tail(dims, q, k_cache, v_cache, page_table, scores, lse_partials, seq_pages, nullptr,
                                    budget_tokens, selected, n_selected, out, lse, workspace, workspace_bytes,
                                    stream);
}

int locks_select_attend_tail(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                             const uint16_t* v_cache, const int32_t* page_table, const float* scores,
                             const float* lse_partials, const int32_t* seq_pages, const int32_t* tail_tokens,
                             int32_t budget_tokens, int32_t* selected, int32_t* n_selected, uint16_t* out,
                             float* lse, void* workspace, size_t workspace_bytes, void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (budget_tokens < 0) return LOCKS_ERR_INVALID_ARG;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !k_cache || !v_cache || !page_table || !scores || !seq_pages || !selected || !n_selected || !out)
        return LOCKS_ERR_INVALID_ARG;
    if (!aligned(q, 8) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return LOCKS_ERR_INVALID_ARG;
    if (lse_partials && !aligned(lse_partials, 16)) return LOCKS_ERR_INVALID_ARG;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    if (!select_fits(dims->max_pages_per_seq, locks::SAMode::kSelectAttend)) return LOCKS_ERR_UNSUPPORTED;
    return select_attend_impl(dims, q, k_cache, v_cache, page_table, scores, lse_partials, seq_pages, tail_tokens,
                              budget_tokens, selected, n_selected, out, lse, workspace,
                              static_cast<cudaStream_t>(stream));
}

int locks_decode_step(const locks_dims_t* dims, const float* q, const uint16_t* k_cache, const uint16_t* v_cache,
                      locks_summaries_t summaries, const int32_t* page_table, const int32_t* seq_pages,
                      int32_t budget_tokens, uint16_t* out, float* lse, float* scores, int32_t* selected,
                      int32_t* n_selected, void* workspace, size_t workspace_bytes, void* stream) {
    return locks_decode_step_tail(dims, q, k_cache, v_cache, summaries, page_table, seq_pages, nullptr,
                                  budget_tokens, out, lse, scores, selected, n_selected, workspace, workspace_bytes,
                                  stream);
}

int locks_decode_step_tail(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                           const uint16_t* v_cache, locks_summaries_t summaries, const int32_t* page_table,
                           const int32_t* seq_pages, const int32_t* tail_tokens, int32_t budget_tokens,
                           uint16_t* out, float* lse, float* scores, int32_t* selected, int32_t* n_selected,
                           void* workspace, size_t workspace_bytes, void* stream) {
    int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    if (budget_tokens < 0) return LOCKS_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(dims, budget_tokens);
    if ((v = check_ws(workspace, workspace_bytes, L.total)) != LOCKS_OK) return v;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !k_cache || !v_cache || !page_table || !seq_pages || !out) return LOCKS_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return LOCKS_ERR_INVALID_ARG;
    if ((v = check_summaries(summaries)) != LOCKS_OK) return v;
    if (!select_fits(dims->max_pages_per_seq, locks::SAMode::kSelectAttend)) return LOCKS_ERR_UNSUPPORTED;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    if (!scores) scores = reinterpret_cast<float*>(base + L.scores);
    if (!selected) selected = reinterpret_cast<int32_t*>(base + L.selected);
    if (!n_selected) n_selected = reinterpret_cast<int32_t*>(base + L.n_selected);
    float* partials = reinterpret_cast<float*>(base + L.partials);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dims->max_pages_per_seq > 0) {
        // with tails, pages are being filled and their one-page builds run on another
        // stream: leave them an SM rather than have one scorer CTA wait for it
        v = score_impl(dims, q, summaries, page_table, seq_pages, scores, partials, workspace, st,
                       tail_tokens ? 1 : 0);
        if (v != LOCKS_OK) return v;
    }
    return select_attend_impl(dims, q, k_cache, v_cache, page_table, scores, partials, seq_pages, tail_tokens,
                              budget_tokens, selected, n_selected, out, lse, workspace, st, tail_tokens ? 1 : 0);
}

int locks_get_device_status(const void* workspace, int32_t* status, void* stream) {
    if (!workspace || !status) return LOCKS_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t host = 0;
    cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof(host), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e);
    *status = host;
    return LOCKS_OK;
}

int locks_clear_device_status(void* workspace, void* stream) {
    if (!workspace) return LOCKS_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)));
}

int locks_selftest_bounded_wait(void* workspace, size_t workspace_bytes, uint64_t limit_ns, void* stream) {
    if (!workspace) return LOCKS_ERR_INVALID_ARG;
    const int v = check_ws(workspace, workspace_bytes, kAlign);
    if (v != LOCKS_OK) return v;
    locks::DeviceStatus st;
    st.word = static_cast<int32_t*>(workspace);
    st.wait_limit_ns = limit_ns == 0 ? 1000000ull : limit_ns;
    return cuda_status(locks::launch_wait_selftest(st, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ------------------------------------------------------------- ablations

namespace {

struct AbLayout {
    size_t moment, q_proj, total;
};
AbLayout ab_layout(const locks_dims_t* d) {
    AbLayout w;
    const size_t B = static_cast<size_t>(d->batch);
    w.moment = kAlign;
    w.q_proj = w.moment + align_up(B * d->num_kv_heads * 128 * 128 * sizeof(float));
    w.total = w.q_proj + align_up(B * d->num_q_heads * 128 * sizeof(float));
    return w;
}

locks::AblationArgs ab_args(const locks_dims_t* d, const float* q, const uint16_t* k_cache,
                            const int32_t* page_table, const int32_t* seq_pages, void* ws) {
    locks::AblationArgs a = {};
    a.q = q;
    a.k_cache = k_cache;
    a.page_table = page_table;
    a.seq_pages = seq_pages;
    a.batch = d->batch;
    a.hq = d->num_q_heads;
    a.hkv = d->num_kv_heads;
    a.max_pages = d->max_pages_per_seq;
    a.num_phys = d->num_phys_pages;
    a.st = status_of(ws);
    return a;
}

// Common checks of the ablation calls; LOCKS_OK means "launch".
int ab_check(const locks_dims_t* d, const uint16_t* k_cache, const int32_t* page_table,
             const int32_t* seq_pages) {
    int v = validate_dims(d);
    if (v != LOCKS_OK) return v;
    if (d->batch > 0 && (!k_cache || !page_table || !seq_pages)) return LOCKS_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16)) return LOCKS_ERR_INVALID_ARG;
    if (static_cast<long>(d->max_pages_per_seq + 127) / 64 > 65535) return LOCKS_ERR_UNSUPPORTED;
    if (current_device() < 0) return LOCKS_ERR_CUDA;
    return LOCKS_OK;
}

bool valid_bits(int32_t b) { return b == 0 || (b >= 2 && b <= 8); }

}  // namespace

extern "C" {

int locks_ablation_workspace_size(const locks_dims_t* dims, size_t* bytes) {
    if (!bytes) return LOCKS_ERR_INVALID_ARG;
    const int v = validate_dims(dims);
    if (v != LOCKS_OK) return v;
    *bytes = ab_layout(dims).total;
    return LOCKS_OK;
}

int locks_exact_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                       const int32_t* page_table, const int32_t* seq_pages, float* scores, void* workspace,
                       size_t workspace_bytes, void* stream) {
    int v = ab_check(dims, k_cache, page_table, seq_pages);
    if (v != LOCKS_OK) return v;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !scores) return LOCKS_ERR_INVALID_ARG;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    locks::AblationArgs a = ab_args(dims, q, k_cache, page_table, seq_pages, workspace);
    a.scores = scores;
    return cuda_status(locks::launch_exact_scores(a, static_cast<cudaStream_t>(stream)));
}

int locks_variant_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                         const int32_t* page_table, const int32_t* seq_pages, int32_t rank, int32_t bits_mu,
                         int32_t bits_v, int32_t bits_c, float* scores, void* workspace, size_t workspace_bytes,
                         void* stream) {
    int v = ab_check(dims, k_cache, page_table, seq_pages);
    if (v != LOCKS_OK) return v;
    if (rank < 1 || rank > 15 || !valid_bits(bits_mu) || !valid_bits(bits_v) || !valid_bits(bits_c))
        return LOCKS_ERR_INVALID_ARG;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !scores) return LOCKS_ERR_INVALID_ARG;
    if (workspace && (v = check_ws(workspace, workspace_bytes, kAlign)) != LOCKS_OK) return v;
    locks::AblationArgs a = ab_args(dims, q, k_cache, page_table, seq_pages, workspace);
    a.scores = scores;
    a.rank = rank;
    a.bits_mu = bits_mu;
    a.bits_v = bits_v;
    a.bits_c = bits_c;
    return cuda_status(locks::launch_variant_scores(a, static_cast<cudaStream_t>(stream)));
}

int locks_shared_basis(const locks_dims_t* dims, const uint16_t* k_cache, const int32_t* page_table,
                       const int32_t* seq_pages, int32_t rank, float* basis, float* eigvals, void* workspace,
                       size_t workspace_bytes, void* stream) {
    int v = ab_check(dims, k_cache, page_table, seq_pages);
    if (v != LOCKS_OK) return v;
    if (rank < 0 || rank > 128) return LOCKS_ERR_INVALID_ARG;
    const AbLayout L = ab_layout(dims);
    if ((v = check_ws(workspace, workspace_bytes, L.total)) != LOCKS_OK) return v;
    if (dims->batch == 0) return LOCKS_OK;
    if (rank > 0 && !basis) return LOCKS_ERR_INVALID_ARG;
    locks::AblationArgs a = ab_args(dims, nullptr, k_cache, page_table, seq_pages, workspace);
    a.rank = rank;
    a.moment = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.moment);
    a.basis = basis;
    a.eigvals = eigvals;
    return cuda_status(locks::launch_shared_basis(a, static_cast<cudaStream_t>(stream)));
}

int locks_shared_scores(const locks_dims_t* dims, const float* q, const uint16_t* k_cache,
                        const int32_t* page_table, const int32_t* seq_pages, const float* basis, int32_t rank,
                        float* scores, void* workspace, size_t workspace_bytes, void* stream) {
    int v = ab_check(dims, k_cache, page_table, seq_pages);
    if (v != LOCKS_OK) return v;
    if (rank < 0 || rank > 128) return LOCKS_ERR_INVALID_ARG;
    const AbLayout L = ab_layout(dims);
    if ((v = check_ws(workspace, workspace_bytes, L.total)) != LOCKS_OK) return v;
    if (dims->batch == 0) return LOCKS_OK;
    if (!q || !scores || (rank > 0 && !basis)) return LOCKS_ERR_INVALID_ARG;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* qp = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + L.q_proj);
    locks::AblationArgs a = ab_args(dims, q, k_cache, page_table, seq_pages, workspace);
    a.rank = rank;
    a.basis = const_cast<float*>(basis);
    a.q_proj = qp;
    if ((v = cuda_status(locks::launch_project_queries(a, st))) != LOCKS_OK) return v;
    a.q = qp;
    a.scores = scores;
    return cuda_status(locks::launch_exact_scores(a, st));
}

}  // extern "C"

namespace locks {

// One thread waits on an mbarrier whose phase nothing completes (expected
// count 2, one arrive); the bounded wait must give up and record a timeout.
__global__ void wait_selftest_kernel(DeviceStatus st) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 2);
        fence_barrier_init();
        mbar_arrive(&bar);
        if (!mbar_wait_bounded(&bar, 0, st.wait_limit_ns)) report_error(st, LOCKS_ERR_TIMEOUT);
    }
}

cudaError_t launch_wait_selftest(DeviceStatus st, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(st);
    return cudaGetLastError();
}

}  // namespace locks
