"""Host-side logic of bench.py that needs no GPU: workload selection and byte accounting."""
import numpy as np

import bench
from continuous_batching_gb300 import workloads as wl


def test_unique_bytes_count_shared_prompt_blocks_once():
    st = wl.make_config("prefix", with_pool=False)
    per_token = 2 * st.Hkv * st.D * 2
    prompts, prompt_tokens = st.notes["prompts"], st.notes["prompt_tokens"]
    own = int((st.ctx_lens.astype(np.int64) - prompt_tokens).sum())
    assert bench.unique_kv_bytes(st) == (prompts * prompt_tokens + own) * per_token
    assert bench.kv_bytes(st) == int(st.ctx_lens.astype(np.int64).sum()) * per_token


def test_unique_bytes_equal_logical_bytes_without_sharing():
    st = wl.make_config("decode", with_pool=False)
    assert bench.unique_kv_bytes(st) == bench.kv_bytes(st)


def test_every_workload_has_a_description_and_seed():
    for name in bench.WORKLOADS:
        if name == "prefill":
            continue
        assert bench.rank_seed(name, 0) == {"decode": 1, "mixed": 2, "longtail": 3,
                                            "prefix": 4, "long16k": 5}[name]
    assert set(bench.TOKEN_WORKLOADS) <= set(bench.WORKLOADS)


def test_cpu_baseline_pool_matches_the_oracle_work_on_the_tiny_step():
    """The multi-core CPU baseline runs the oracle in spawned workers over shared memory and
    counts whole passes: two workers, a zero budget (one pass)."""
    st = wl.make_config("tiny")
    r = bench.cpu_baseline(st, budget_s=0.0, workers=2)
    assert r["cores"] == 2 and r["kind"] == "oracle" and r["value"] > 0
    assert "1 full pass" in r["sample"]
    t = bench.cpu_baseline(st, budget_s=0.0, tokens=True, workers=2)
    assert t["unit"] == "tokens/s" and t["value"] > 0
