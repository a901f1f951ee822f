// Cache-aware scheduling over the radix tree: a round-based simulation of a
// serving loop that reports per-request admission, cache hits and finish
// rounds, and the prefill work the cache saved.
//
// Sources (page title, section):
//  * "SGLang：从前端 DSL 到 SRT 服务运行时", section "用基数树实现前缀复用":
//    cache-aware scheduling serves the waiting request with the longest
//    cached prefix first (an approximate depth-first walk of the tree);
//    leaf-first LRU eviction; reference counts protect running requests.
//  * The CS349D lecture-16 notes, §3.1-3.3: a runtime with continuous
//    batching (every request past prefill decodes one token per round), a
//    per-round prefill token budget (chunked prefill), FCFS or longest-prefix
//    -first queueing that defers a request whose uncached prefix largely
//    coincides with one admitted in the same round, and insertion of the
//    prompt into the tree at prefill completion rather than at request end.
//
// The round structure, allocation at admission and the defer rule's exact
// form are readings of those descriptions: a round takes arrivals, queue
// ordering, admission, prefill within the budget, one decode token per
// request past prefill, then finishing; admission allocates the uncached
// prompt and the whole output at once; "largely coincides" compares the next
// defer_tokens uncached prompt tokens of requests with equal cached length.

#include <algorithm>
#include <cstring>
#include <vector>

#include "sglattn.h"

namespace {

struct Req {
    const sgl_sim_request* in;
    int64_t arrive = -1;          // known once its dependency has finished
    bool queued = false, running = false, done = false;
    int64_t cached = 0, remaining = 0, generated = 0;
    bool prefilled = false;
    int64_t prefill_round = -1;
    sgl_node lock = 0;            // node this request holds a reference on
    std::vector<int32_t> row;     // slots of prompt + output
    std::vector<int32_t> seq;     // prompt + output tokens
};

}  // namespace

extern "C" {

int sgl_sim_run(sgl_tree* tree, const sgl_sim_config* cfg, int32_t n, const sgl_sim_request* reqs,
                sgl_sim_result* per_req, sgl_sim_stats* stats) {
    if (!tree || !cfg || n < 0 || (n > 0 && (!reqs || !per_req)) || !stats) return SGL_ERR_INVALID_ARG;
    if (cfg->prefill_budget < 1 || cfg->max_running < 1 || cfg->defer_tokens < 0 || cfg->max_rounds < 1 ||
        (cfg->policy != SGL_SCHED_FCFS && cfg->policy != SGL_SCHED_LPM) ||
        (cfg->insert_at != SGL_INSERT_AT_PREFILL && cfg->insert_at != SGL_INSERT_AT_FINISH))
        return SGL_ERR_INVALID_ARG;
    std::vector<Req> R(n);
    for (int32_t i = 0; i < n; ++i) {
        const sgl_sim_request& q = reqs[i];
        if (q.prompt_len < 1 || q.output_len < 1 || !q.prompt || !q.output || q.depends_on >= i ||
            q.depends_on < -1 || q.delay < 0 || (q.depends_on < 0 && q.arrive_round < 0))
            return SGL_ERR_INVALID_ARG;
        R[i].in = &q;
        R[i].arrive = q.depends_on < 0 ? q.arrive_round : -1;
        R[i].seq.assign(q.prompt, q.prompt + q.prompt_len);
        R[i].seq.insert(R[i].seq.end(), q.output, q.output + q.output_len);
        per_req[i] = sgl_sim_result{-1, -1, 0, -1, -1};
    }
    std::memset(stats, 0, sizeof(*stats));
    std::vector<int32_t> waiting, running;   // request indices
    std::vector<int32_t> scratch;
    auto tree_tokens = [&]() {
        sgl_tree_stats_t ts;
        sgl_tree_stats(tree, &ts);
        return ts.tree_tokens;
    };
    auto match_len = [&](const Req& r, sgl_node* node, std::vector<int32_t>* slots) {
        int64_t m = 0;
        slots->assign(r.in->prompt_len, 0);
        sgl_tree_match(tree, r.in->prompt, r.in->prompt_len, &m, slots->data(), node);
        slots->resize(m);
        return m;
    };
    int32_t finished = 0;
    int64_t round = 0;
    for (; finished < n; ++round) {
        if (round >= cfg->max_rounds) return SGL_ERR_STATE;
        // 1. arrivals, in (arrival round, index) order
        std::vector<int32_t> arriving;
        for (int32_t i = 0; i < n; ++i)
            if (!R[i].queued && R[i].arrive >= 0 && R[i].arrive <= round) arriving.push_back(i);
        std::stable_sort(arriving.begin(), arriving.end(),
                         [&](int32_t a, int32_t b) { return R[a].arrive < R[b].arrive; });
        for (int32_t i : arriving) {
            R[i].queued = true;
            per_req[i].arrive_round = R[i].arrive;
            waiting.push_back(i);
        }
        // 2. order the waiting queue
        std::vector<int32_t> order = waiting;
        if (cfg->policy == SGL_SCHED_LPM) {
            std::vector<std::pair<int64_t, int32_t>> key;
            for (int32_t i : order) {
                sgl_node nd;
                key.push_back({match_len(R[i], &nd, &scratch), i});
            }
            std::vector<int64_t> pos(n, 0);
            for (size_t k = 0; k < order.size(); ++k) pos[order[k]] = (int64_t)k;
            std::stable_sort(key.begin(), key.end(), [&](const std::pair<int64_t, int32_t>& a,
                                                         const std::pair<int64_t, int32_t>& b) {
                return a.first > b.first;
            });
            for (size_t k = 0; k < key.size(); ++k) order[k] = key[k].second;
        }
        // 3. admission
        std::vector<int32_t> admitted_now;
        for (int32_t i : order) {
            if ((int32_t)running.size() >= cfg->max_running) break;
            Req& r = R[i];
            sgl_node mnode = 0;
            std::vector<int32_t> mslots;
            const int64_t m = match_len(r, &mnode, &mslots);
            if (cfg->policy == SGL_SCHED_LPM && cfg->defer_tokens > 0) {
                const int64_t k = std::min<int64_t>(cfg->defer_tokens, r.in->prompt_len - m);
                bool defer = false;
                for (int32_t j : admitted_now) {
                    const Req& o = R[j];
                    if (o.cached == m && k > 0 && o.in->prompt_len >= m + k &&
                        std::equal(r.in->prompt + m, r.in->prompt + m + k, o.in->prompt + m)) {
                        defer = true;
                        break;
                    }
                }
                if (defer) continue;
            }
            sgl_tree_lock(tree, mnode);
            const int64_t need = (int64_t)r.seq.size() - m;
            std::vector<int32_t> fresh(need);
            const int64_t before = tree_tokens();
            const int st = sgl_tree_alloc(tree, need, fresh.data());
            stats->evicted_tokens += before - tree_tokens();
            if (st != SGL_OK) {
                sgl_tree_unlock(tree, mnode);
                if (st != SGL_ERR_NO_SLOTS) return st;
                break;   // the pool is full: no more admissions this round
            }
            r.lock = mnode;
            r.cached = m;
            r.remaining = r.in->prompt_len - m;
            r.row = mslots;
            r.row.insert(r.row.end(), fresh.begin(), fresh.end());
            r.running = true;
            per_req[i].admit_round = round;
            per_req[i].cached_tokens = m;
            stats->prompt_tokens += r.in->prompt_len;
            stats->cached_tokens += m;
            admitted_now.push_back(i);
            running.push_back(i);
            waiting.erase(std::find(waiting.begin(), waiting.end(), i));
        }
        // 4. prefill within the round's token budget, in admission order
        int64_t budget = cfg->prefill_budget;
        for (int32_t i : running) {
            Req& r = R[i];
            if (r.prefilled || budget == 0) continue;
            const int64_t t = std::min(r.remaining, budget);
            r.remaining -= t;
            budget -= t;
            stats->prefill_tokens += t;
            if (r.remaining == 0) {
                r.prefilled = true;
                r.prefill_round = round;
                per_req[i].prefill_done_round = round;
                if (cfg->insert_at == SGL_INSERT_AT_PREFILL) {
                    int64_t dup = 0;
                    sgl_node last = 0;
                    const int64_t P_full = r.in->prompt_len;
                    sgl_tree_insert(tree, r.in->prompt, r.row.data(), P_full, &dup, &last);
                    sgl_tree_lock(tree, last);
                    sgl_tree_unlock(tree, r.lock);
                    r.lock = last;
                }
            }
        }
        // 5. decode: one token per request whose prefill finished in an earlier round
        std::vector<int32_t> still;
        for (int32_t i : running) {
            Req& r = R[i];
            if (r.prefilled && r.prefill_round < round) {
                ++r.generated;
                ++stats->decode_tokens;
            }
            if (r.prefilled && r.generated == r.in->output_len) {
                // finish: the whole sequence into the tree, references released,
                // a partial tail page freed
                int64_t dup = 0;
                sgl_node last = 0;
                sgl_tree_insert(tree, r.seq.data(), r.row.data(), (int64_t)r.seq.size(), &dup, &last);
                sgl_tree_unlock(tree, r.lock);
                sgl_tree_lock(tree, last);
                sgl_tree_finish(tree, last, r.row.data(), (int64_t)r.seq.size());
                r.running = false;
                r.done = true;
                per_req[i].finish_round = round;
                ++finished;
                for (int32_t j = i + 1; j < n; ++j)
                    if (R[j].in->depends_on == i) R[j].arrive = round + R[j].in->delay;
            } else {
                still.push_back(i);
            }
        }
        running.swap(still);
    }
    stats->rounds = round;
    return SGL_OK;
}

}  // extern "C"
