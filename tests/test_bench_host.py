"""Host logic of the benchmark, on CPU: the whole-job aggregation over ranks
(world size 2 over gloo, as torchrun launches the replicas) and the
algorithmic byte counts the roofline divides by."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        # rank r processed 100 (r + 1) units in 0.5 + r seconds
        units, secs = bench.aggregate(100.0 * (rank + 1), 0.5 + rank, world)
        bench.barrier(world)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{units} {secs}\n")
    finally:
        dist.destroy_process_group()


def test_aggregate_two_ranks_gloo(tmp_path):
    """Units are summed over the ranks, time is the slowest rank's, and every
    rank sees the same whole-job numbers."""
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for r in range(world):
        units, secs = map(float, open(tmp_path / f"rank{r}.txt").read().split())
        assert units == 300.0
        assert secs == 1.5


def test_aggregate_single_rank_is_identity():
    assert bench.aggregate(48.0, 0.25, 1) == (48.0, 0.25)


def _llama():
    return dict(M=8, d=4096, r=512, V=128256, T=0.0, gamma=6, B=8, u_full=None)


def test_head_bytes_are_w_up_plus_z():
    """One up-projection launch must move W_up (V x r bf16) and the z rows
    (M x r bf16) once: 131,342,336 bytes at the Llama shape."""
    x = _llama()
    kb = bench.kernel_bytes(x, 0.0, 0)
    assert kb["k_head_mma"] == 128256 * 512 * 2 + 8 * 512 * 2 == 131342336
    assert kb["k_head_stream"] == kb["k_head_mma"]
    assert kb["k_down_proj"] == 512 * 4096 * 2 + 8 * 4096 * 2 + 8 * 512 * 2
    assert "k_gather_logits" not in kb


def test_verify_rows_needed():
    """Rows the accept chain needs: positions 0..n of the target rows (n
    accepted), plus, when sampling, the draft rows of the drafted positions
    among them."""
    acc = torch.tensor([0, 2, 6, 1], dtype=torch.int32)
    x = dict(_llama(), gamma=6)
    assert bench.verify_rows_read(x, acc) == 1 + 3 + 7 + 2
    xs = dict(x, T=1.0)
    assert bench.verify_rows_read(xs, acc) == (1 + 3 + 7 + 2) + (1 + 3 + 6 + 2)
    # the low-rank verifier reads no draft rows
    assert bench.verify_rows_read(dict(xs, lowrank=True), acc) == 1 + 3 + 7 + 2
    kb = bench.kernel_bytes(x, 0.0, 13)
    assert kb["k_verify_rows"] == 13 * 128256 * 4


def test_specvocab_gather_bytes():
    x = dict(M=32, d=4096, r=256, V=151936, T=1.0, gamma=6, B=32, u_full=object())
    kb = bench.kernel_bytes(x, 50000.0, 0)
    assert kb["k_gather_logits"] == 50000 * 4096 * 2 + 32 * 4096 * 2
    assert kb["k_topk"] == 32 * 151936 * 4


def test_quantiles_nearest_rank():
    v = list(range(11))            # 0 .. 10
    assert bench.quantiles(v, (0.1, 0.5, 0.9)) == [1, 5, 9]
    assert bench.quantiles([3.0], (0.1, 0.5, 0.9)) == [3.0, 3.0, 3.0]
    assert bench.quantiles([5, 1, 3], (0.0, 1.0)) == [1, 5]


def test_timeline_exclusive_times_add_up_to_busy_time():
    """Overlapping launches (a dependent launch starting before its
    predecessor ends) are charged only past the latest end before them, so a
    replay's exclusive times sum to its busy time, never to more."""
    from speculative_decoding_drafter_slimspec_gb300 import timeline
    recs = [("k_a", 0, 100), ("k_b", 80, 130), ("k_c", 90, 120), ("k_d", 150, 160)]
    excl, busy = timeline.exclusive_times(recs)
    assert excl == [100, 30, 0, 10]
    assert busy == 140 <= 160


def test_timeline_summary_per_kernel():
    from speculative_decoding_drafter_slimspec_gb300 import timeline
    one = [("k_head_mma", 0, 100), ("k_head_mma_finish", 90, 110), ("k_verify_rows", 120, 150)]
    recs = one + [(k, s + 1000, e + 1000) for k, s, e in one] + [("other", 5, 6)]
    out = timeline.summarize(recs, per_replay=3)
    assert out["replays"] == 2
    k = out["kernels"]
    assert k["k_head_mma"]["us_per_launch"] == 0.1
    assert k["k_head_mma_finish"]["exclusive_us_per_step"] == 0.01
    assert abs(sum(v["share"] for v in k.values()) - 1.0) < 1e-12
    assert out["busy_us"] == 0.14 and out["wall_us"] == 0.15


def test_kernel_kind_from_mangled_names():
    from speculative_decoding_drafter_slimspec_gb300 import timeline
    assert timeline.kernel_kind("_ZN2ss10k_head_mmaILb0ELi0ELb1EEEvPKt") == "k_head_mma"
    assert timeline.kernel_kind("_ZN2ss15k_verify_decideILb0EEEvPKf") == "k_verify_decide"
    assert timeline.kernel_kind("void ss::k_topk(float const*, int)") == "k_topk"


def test_head_call_and_verify_bytes():
    x = _llama()
    assert bench.head_call_bytes(x) == 128256 * 512 * 2 + 512 * 4096 * 2 + 8 * 4096 * 2 + 8 * 4
    assert bench.verify_all_bytes(x) == 8 * 7 * 128256 * 4 + 8 * 6 * 4
    xs = dict(x, T=1.0)
    assert bench.verify_all_bytes(xs) == 8 * 7 * 128256 * 4 + 8 * 6 * 128256 * 4 + 8 * 6 * 4
