// Host step scheduler: builds the flat ragged step that paged_attention_step consumes.
//
// "P3: native paged-KV continuous-batching sampler", Design / engine.py:
//   - every sequence is tokens + num_computed; a step schedules n_new = min(remaining, chunk,
//     budget) per sequence; prefill, chunked prefill, decode and recompute after preemption
//     are one path; a sequence samples when its scheduled tokens reach the end of its tokens;
//     decodes are scheduled first; prefill chunks and decodes share one flat ragged step;
//   - FIFO admission if the whole current token list fits; on block exhaustion the youngest
//     unscheduled running sequence is preempted by recompute (blocks freed, num_computed = 0,
//     tokens kept);
//   - prefix sharing: a waiting sequence adopts the leading full blocks of a running one,
//     defers while the leader is still computing them, and recomputes its last prompt token.
// The points the page leaves open are fixed as follows:
//   - remaining = tokens - num_computed; a decode is a running sequence with remaining 1;
//   - running sequences are visited decodes first, then the rest, each in admission order,
//     then waiting sequences are admitted in order while budget remains; admission stops at
//     the first one that does not fit or defers;
//   - a running sequence grows with ensure_capacity(num_computed + n_new); on exhaustion the
//     youngest running sequence not yet scheduled this step (other than itself) is preempted
//     and the attempt repeats; with none left it sits this step out;
//   - admission reserves blocks for the whole current token list, all or nothing;
//   - a preempted sequence goes back to the head of the waiting queue;
//   - a follower shares (prompt - 1) / block_size full blocks of its leader once the leader
//     has computed them, defers while the leader waits or computes, and is admitted without
//     sharing when the leader has finished; it then starts at the first unshared position;
//   - after a step every scheduled sequence adds n_new to num_computed; one that reaches the
//     end of its tokens samples: at max_new it finishes (blocks freed), else it gains a token.
#include <algorithm>
#include <cstdint>
#include <deque>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "common.h"

namespace {

struct SeqState {
    int32_t n_tokens = 0;       // prompt + sampled so far
    int32_t prompt_len = 0;
    int32_t num_computed = 0;   // tokens whose K/V are in the cache
    int32_t max_new = 0;
    int32_t generated = 0;
    int32_t leader = -1;
    int64_t stamp = -1;         // admission order of the current residency
    bool finished = false;
};

}  // namespace

struct pa_scheduler {
    pa_allocator* alloc = nullptr;
    int32_t block_size = 0, chunk = 0, budget = 0;
    std::unordered_map<int32_t, SeqState> seqs;
    std::deque<int32_t> waiting;
    std::vector<int32_t> running;                        // admission order
    std::vector<std::pair<int32_t, int32_t>> scheduled;  // (seq, n_new) of the pending step
    bool pending = false;
    int64_t next_stamp = 0;
    int64_t preemptions = 0;
};

namespace {

int32_t remaining(const SeqState& s) { return s.n_tokens - s.num_computed; }

void preempt(pa_scheduler* S, int32_t q) {
    pa_alloc_free_seq(S->alloc, q);
    S->running.erase(std::find(S->running.begin(), S->running.end(), q));
    SeqState& s = S->seqs[q];
    s.num_computed = 0;
    s.stamp = -1;
    S->waiting.push_front(q);
    ++S->preemptions;
}

bool is_running(const pa_scheduler* S, int32_t q) {
    return std::find(S->running.begin(), S->running.end(), q) != S->running.end();
}

}  // namespace

extern "C" {

int32_t pa_sched_create(int32_t num_blocks, int32_t block_size, int32_t chunk, int32_t budget,
                        pa_scheduler** out) {
    if (!out || num_blocks < 0 || block_size <= 0 || chunk <= 0 || budget <= 0)
        return PA_ERR_INVALID;
    pa_allocator* a = nullptr;
    const int32_t st = pa_alloc_create(num_blocks, block_size, &a);
    if (st) return st;
    auto* S = new pa_scheduler;
    S->alloc = a;
    S->block_size = block_size;
    S->chunk = chunk;
    S->budget = budget;
    *out = S;
    return PA_OK;
}

int32_t pa_sched_destroy(pa_scheduler* S) {
    if (S) pa_alloc_destroy(S->alloc);
    delete S;
    return PA_OK;
}

pa_allocator* pa_sched_allocator(pa_scheduler* S) { return S ? S->alloc : nullptr; }

int32_t pa_sched_add(pa_scheduler* S, int32_t seq, int32_t prompt_len, int32_t max_new,
                     int32_t leader) {
    if (!S || seq < 0 || prompt_len < 1 || max_new < 1 || leader < -1) return PA_ERR_INVALID;
    if (S->seqs.count(seq)) return PA_ERR_STATE;
    SeqState s;
    s.n_tokens = prompt_len;
    s.prompt_len = prompt_len;
    s.max_new = max_new;
    s.leader = leader;
    S->seqs.emplace(seq, s);
    S->waiting.push_back(seq);
    return PA_OK;
}

int32_t pa_sched_step(pa_scheduler* S, int32_t* seqs, int32_t* n_new, int32_t* ctx_lens,
                      int32_t cap, int32_t* n_out) {
    if (!S || !n_out || cap < 0) return PA_ERR_INVALID;
    if (S->pending) return PA_ERR_STATE;
    const size_t live = S->running.size() + S->waiting.size();
    if (size_t(cap) < live || (live > 0 && (!seqs || !n_new || !ctx_lens))) return PA_ERR_INVALID;
    int32_t budget = S->budget;
    std::unordered_set<int32_t> done;
    std::vector<std::pair<int32_t, int32_t>> out;
    std::vector<int32_t> order;
    for (int32_t q : S->running)
        if (remaining(S->seqs[q]) == 1) order.push_back(q);
    for (int32_t q : S->running)
        if (remaining(S->seqs[q]) > 1) order.push_back(q);
    for (int32_t q : order) {
        if (budget == 0) break;
        if (!is_running(S, q)) continue;              // preempted earlier in this step
        SeqState& s = S->seqs[q];
        const int32_t n = std::min({remaining(s), S->chunk, budget});
        bool ok = false;
        for (;;) {
            const int32_t st = pa_alloc_ensure_capacity(S->alloc, q, s.num_computed + n);
            if (st == PA_OK) {
                ok = true;
                break;
            }
            if (st != PA_ERR_OOM) return st;
            int32_t victim = -1;
            int64_t best = -1;
            for (int32_t v : S->running)
                if (v != q && !done.count(v) && S->seqs[v].stamp > best) {
                    best = S->seqs[v].stamp;
                    victim = v;
                }
            if (victim < 0) break;
            preempt(S, victim);
        }
        if (ok) {
            out.emplace_back(q, n);
            done.insert(q);
            budget -= n;
        }
    }
    while (!S->waiting.empty() && budget > 0) {
        const int32_t q = S->waiting.front();
        SeqState& s = S->seqs[q];
        int32_t n_shared = 0, src = -1;
        if (s.leader >= 0 && S->seqs.count(s.leader)) {
            const SeqState& lead = S->seqs[s.leader];
            int32_t share = (s.prompt_len - 1) / S->block_size;
            if (lead.finished) {
                share = 0;
            } else if (!is_running(S, s.leader) ||
                       int64_t(lead.num_computed) < int64_t(share) * S->block_size) {
                break;                                   // defers while the leader computes
            }
            if (share > 0) {
                n_shared = share;
                src = s.leader;
            }
        }
        const int32_t st = pa_alloc_admit(S->alloc, q, s.n_tokens, src, n_shared);
        if (st == PA_ERR_OOM) break;
        if (st) return st;
        S->waiting.pop_front();
        S->running.push_back(q);
        s.stamp = S->next_stamp++;
        s.num_computed = n_shared * S->block_size;
        const int32_t n = std::min({remaining(s), S->chunk, budget});
        out.emplace_back(q, n);
        done.insert(q);
        budget -= n;
    }
    for (size_t i = 0; i < out.size(); ++i) {
        const SeqState& s = S->seqs[out[i].first];
        seqs[i] = out[i].first;
        n_new[i] = out[i].second;
        ctx_lens[i] = s.num_computed + out[i].second;
    }
    *n_out = int32_t(out.size());
    S->scheduled = std::move(out);
    S->pending = true;
    return PA_OK;
}

int32_t pa_sched_commit(pa_scheduler* S, int32_t* finished, int32_t cap, int32_t* n_finished) {
    if (!S || !n_finished || cap < 0) return PA_ERR_INVALID;
    if (!S->pending) return PA_ERR_STATE;
    if (size_t(cap) < S->scheduled.size() || (cap > 0 && !finished)) return PA_ERR_INVALID;
    int32_t k = 0;
    for (const auto& e : S->scheduled) {
        SeqState& s = S->seqs[e.first];
        s.num_computed += e.second;
        if (s.num_computed != s.n_tokens) continue;
        s.generated += 1;
        if (s.generated == s.max_new) {
            pa_alloc_free_seq(S->alloc, e.first);
            S->running.erase(std::find(S->running.begin(), S->running.end(), e.first));
            s.finished = true;
            finished[k++] = e.first;
        } else {
            s.n_tokens += 1;
        }
    }
    *n_finished = k;
    S->scheduled.clear();
    S->pending = false;
    return PA_OK;
}

int32_t pa_sched_counts(const pa_scheduler* S, int32_t* n_waiting, int32_t* n_running,
                        int64_t* preemptions) {
    if (!S) return PA_ERR_INVALID;
    if (n_waiting) *n_waiting = int32_t(S->waiting.size());
    if (n_running) *n_running = int32_t(S->running.size());
    if (preemptions) *preemptions = S->preemptions;
    return PA_OK;
}

int32_t pa_sched_seq(const pa_scheduler* S, int32_t seq, int32_t* n_tokens,
                     int32_t* num_computed, int32_t* generated) {
    if (!S) return PA_ERR_INVALID;
    auto it = S->seqs.find(seq);
    if (it == S->seqs.end()) return PA_ERR_STATE;
    if (n_tokens) *n_tokens = it->second.n_tokens;
    if (num_computed) *num_computed = it->second.num_computed;
    if (generated) *generated = it->second.generated;
    return PA_OK;
}

}  // extern "C"
