"""Host logic of bench.py, checked without a GPU.

- The analytic HBM bytes per window, against the closed forms worked out by hand.
- The multi-rank timing path: two gloo ranks on the CPU take the max over ranks,
  the way torchrun replicas do on GPUs.
- The CPU baseline's threaded oracle sample and the reference arm.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def test_window_bytes_of_the_layer_workload():
    s = synth.PRESETS["mamba2_layer_b256_l16"]
    S = 4 * 128 * 64 * 128
    r = 4 * 128 + 2 * 128 * 64 + 2 * 8 * 128
    assert (S, r) == (4194304, 18944)
    inp, out = r + 2 * 8 * 128, 4 * 128 * 64
    expect = 16 * S + S + r * 16 * 15 // 2 + 16 * (inp + out) + 15 * r
    wb = bench.window_bytes(s)
    assert wb["replay_window"] == expect == 74720768
    assert wb["replay_per_seq_step"] == 4670048
    assert wb["conventional_per_seq_step"] == 2 * S + inp + out == 8442368
    # read copies: (L-1) non-flush reads of the copy, one flush read of S and one write of S + copy
    c4 = 128 * (64 * 128 + 4 * 64)
    e4 = bench.window_bytes(s, "e4m3")["replay_window"]
    assert e4 == 15 * c4 + S + S + c4 + r * 120 + 16 * (inp + out) + 15 * r
    assert bench.copy_bytes_per_head(s, "e2m1") == 64 * 64 + 64 * 8 + 64 * 4


def _free_port():
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        results[rank] = bench.max_over_ranks(float(10 * (rank + 1)), world)
    finally:
        dist.destroy_process_group()


def test_window_bytes_of_a_delta_rule_layer():
    """Delta-rule windows: the inputs carry beta (4 B per head) and the buffered
    records hold fp32 pseudo-values instead of bf16 values (2 more bytes per
    element), for the 120 buffered-record reads and 15 appends of a window."""
    s = synth.PRESETS["mamba2_layer_b256_l16"]
    outer, delta = bench.window_bytes(s), bench.window_bytes(s, delta=True)
    beta_in = 16 * 4 * 128                      # one beta per head and step
    ring_extra = (16 * 15 // 2 + 15) * 2 * 128 * 64  # record reads + appends, 2 B more per element
    assert delta["replay_window"] - outer["replay_window"] == beta_in + ring_extra == 2220032
    assert delta["state"] == outer["state"]
    assert delta["replay_per_seq_step"] == 4808800


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    results = mp.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
    assert dict(results) == {0: 20.0, 1: 20.0}


def _reference_rank(rank, world, port, results):
    import contextlib
    import io
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world))
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        bench.main(["--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "3"])
    results[rank] = out.getvalue()


def test_reference_arm_under_two_gloo_ranks():
    """Launched as torchrun replicas, the reference arm runs on rank 0 alone, which prints
    the one JSON line (n_gpus = world size); the other rank prints nothing and exits."""
    import json
    world = 2
    results = mp.Manager().dict()
    mp.start_processes(_reference_rank, args=(world, _free_port(), results), nprocs=world, start_method="spawn")
    assert results[1] == ""
    lines = results[0].strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == world and line["value"] > 0


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_runs_on_cpu(capsys):
    """The reference arm (the float64 oracle) prints one JSON line with its own e2e and cpu_baseline."""
    import json
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    if not torch.cuda.is_available():
        with pytest.raises(SystemExit):
            bench.main(["--steps", "1", "--warmup", "3"])


def test_oracle_sample_threads_step_their_own_groups():
    """The CPU baseline's threads each step their own seeded group: the states they
    reach equal a plain sequential run of the same groups, over two calls."""
    import numpy as np

    import oracle
    s = synth.PRESETS["tiny_b2_h2_p16_n16_l4"]
    sample = bench.OracleSample(s, n_seq=2, threads=3, seed=5)
    sample.run(3)
    sample.run(2)
    assert sample.units(5) == 3 * 2 * 5 and sample.done == 5
    sub = s.with_(B=2)
    for t, (S_thread, _) in enumerate(sample.parts):
        gen = synth.make_generator(5 + 7919 * t)
        S = oracle.to_f64(synth.initial_state(sub, gen))
        steps = [tuple(oracle.to_f64(x) for x in synth.decode_step_inputs(sub, gen)) for _ in range(4)]
        for i in range(5):
            S, _ = oracle.conventional_step(S, *steps[i % 4])
        assert np.array_equal(S_thread, S), t


def test_verify_round_bytes_of_the_verify_workload():
    """Verify-round byte model on four sequences of the B=512 T=4 workload's shape,
    with the numbers worked out by hand: a 4 MiB checkpoint, 18,944-byte records,
    20,992 bytes of draft inputs (a record plus its bf16 query) and 32,768-byte
    outputs per sequence."""
    import numpy as np
    s = synth.PRESETS["mamba2_verify_b512_t4"].with_(B=4)
    counts, accepted = np.array([0, 5, 15, 12]), np.array([4, 0, 1, 4])
    vb, fb, after = bench.verify_round_bytes(s, 4, counts, accepted)
    # each sequence: checkpoint once, its committed records, and per draft its inputs,
    # its appended record and its output: 4194304 + c*18944 + 4*(20992 + 18944 + 32768)
    assert vb == 4 * 4194304 + 32 * 18944 + 4 * 4 * 72704 == 18_546_688
    # commit leaves 4, 5, 16, 16 records; the last two fold (read and write the
    # checkpoint, read 16 records); commit moves 12 bytes per sequence
    assert after.tolist() == [4, 5, 0, 0]
    assert fb == 2 * (2 * 4194304 + 16 * 18944) + 12 * 4 == 17_383_472


def test_verify_round_bytes_of_a_delta_rule_layer():
    """The same four sequences as a gated delta-rule layer, worked out by hand: a ring
    record holds alpha (512 B), the fp32 pseudo-value w (32,768 B) and the bf16 key
    (2,048 B), 35,328 bytes; a draft's inputs are alpha and beta (512 B each), v (16,384 B),
    k and q (2,048 B each), 21,504 bytes."""
    import numpy as np
    s = synth.PRESETS["mamba2_verify_b512_t4"].with_(B=4)
    counts, accepted = np.array([0, 5, 15, 12]), np.array([4, 0, 1, 4])
    vb, fb, after = bench.verify_round_bytes(s, 4, counts, accepted, delta=True)
    assert vb == 4 * 4194304 + 32 * 35328 + 4 * 4 * (21504 + 35328 + 32768) == 19_341_312
    assert after.tolist() == [4, 5, 0, 0]
    assert fb == 2 * (2 * 4194304 + 16 * 35328) + 12 * 4 == 17_907_760


def test_window_bytes_with_read_copies():
    """Read-copy windows of the B=256 L=16 layer, worked out by hand. A head's E4M3
    copy is 64 x 128 codes + 64 fp32 row scales = 8,448 B; an E2M1 copy is 4,096 B
    of codes + 512 block scales + 256 B of row scales = 4,864 B. The 15 non-flush
    steps read the copy; the flush step reads and writes the 4 MiB checkpoint and
    writes the copy; records, inputs and outputs are as without a copy:
    120 buffered-record reads and 15 appends of 18,944 B, 16 x (20,992 + 32,768)."""
    s = synth.PRESETS["mamba2_layer_b256_l16"]
    rest = 2 * 4194304 + 135 * 18944 + 16 * (20992 + 32768)
    e4 = bench.window_bytes(s, "e4m3")
    assert e4["replay_window"] == 16 * 128 * 8448 + rest == 29_107_712
    assert e4["replay_per_seq_step"] == 1_819_232
    e2 = bench.window_bytes(s, "e2m1")
    assert e2["replay_window"] == 16 * 128 * 4864 + rest == 21_767_680
    assert e2["replay_per_seq_step"] == 1_360_480


def test_window_bytes_with_an_fp16_checkpoint():
    """FP16 checkpoint (2 MiB per sequence): 16 reads and one write of it per window,
    the same records, inputs and outputs as the FP32 layer."""
    s = synth.PRESETS["mamba2_layer_b256_l16"]
    wb = bench.window_bytes(s, None, ckpt_bytes=2)
    assert wb["replay_window"] == 17 * 2097152 + 135 * 18944 + 16 * (20992 + 32768) == 39_069_184
    assert wb["replay_per_seq_step"] == 2_441_824
