"""Host-side pieces of bench.py that run without a GPU: the oracle baselines
reported beside the importance pass and the rotary embedding."""
import bench


def test_oracle_baselines_of_the_steps_around_verification():
    import workloads as W

    w = W.make_workload("sparse", seed=0, B=2, L_lo=2000, L_hi=3000)
    fn, nbytes, desc = bench.scoring_oracle_sample(w, n_seq=2)
    r = bench.oracle_rate(fn, nbytes, desc, target_s=0.1, max_reps=2)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1
    fn, nbytes, desc = bench.rope_oracle_sample(B=2)
    assert nbytes == 2 * 2 * 16 * (32 + 8) * 128 * 2
    r = bench.oracle_rate(fn, nbytes, desc, target_s=0.1, max_reps=2)
    assert r["value"] > 0 and "paged" in r["sample"]
