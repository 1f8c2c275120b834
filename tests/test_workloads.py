"""The seeded input generators (no GPU): shapes, determinism and the length recipes."""
import numpy as np
import torch

from workloads import CONFIGS, algorithmic_bytes, draw_seq_lens, make_case


def test_generators_are_deterministic():
    a = make_case("tiny")
    b = make_case("tiny")
    for name in ("q", "k_cache", "v_cache", "block_table", "seq_lens"):
        assert torch.equal(getattr(a, name).view(torch.int16) if getattr(a, name).dtype == torch.bfloat16
                           else getattr(a, name),
                           getattr(b, name).view(torch.int16) if getattr(b, name).dtype == torch.bfloat16
                           else getattr(b, name))


def test_tiny_shapes_and_pool():
    c = make_case("tiny")
    assert c.q.shape == (1, 8, 64) and c.k_cache.shape == (64, 16, 2, 64)
    assert int(c.seq_lens[0]) == 256 and c.max_pages == 16
    ids = c.block_table[0].numpy()
    assert len(set(ids.tolist())) == 16 and ids.min() >= 0 and ids.max() < 64
    assert c.scale == np.float32(1 / 8)


def test_length_recipes():
    lens = draw_seq_lens(CONFIGS["batch"]["lens"], 8, 16, 1)
    assert lens.min() >= 1024 and lens.max() <= 4096
    r = draw_seq_lens(CONFIGS["ragged"]["lens"], 64, 16, 2)
    assert r.min() >= 17 and r.max() <= 32768
    assert all(r[i] % 16 != 0 for i in range(0, 64, 4))
    assert 1024 <= np.median(r) <= 4096


def test_pages_are_disjoint_and_poison_marks_padding():
    c = make_case(dict(B=3, Hq=4, Hkv=2, D=16, P=8, lens=("list", [9, 16, 1]), seed=3), poison=True)
    bt = c.block_table.numpy()
    used = [bt[b, j] for b, L in enumerate([9, 16, 1]) for j in range((L + 7) // 8)]
    assert len(used) == len(set(used))
    # slot 1.. of the last page of sequence 0 (9 tokens) is padding -> NaN
    assert torch.isnan(c.k_cache[bt[0, 1], 1:].float()).all()
    assert not torch.isnan(c.k_cache[bt[0, 1], 0].float()).any()
    assert bt[2, 1] in (-1, 1 << 30)


def test_algorithmic_bytes_tiny():
    c = make_case("tiny")
    ab = algorithmic_bytes(c)
    assert ab["kv"] == 2 * 256 * 2 * 64 * 2
    assert ab["total"] == ab["kv"] + 2 * 8 * 64 * 2 + 8 * 4 + 16 * 4 + 4
    assert ab["tail_bytes"] == 0


def test_profile_summaries_agree_with_the_workloads():
    """Every committed ncu summary of the decode kernel names the algorithmic bytes the workload
    definition gives (recomputed here from the seeded lengths), and its DRAM traffic lies between
    those bytes and 4% above them (every K/V byte read once)."""
    import glob
    import os
    import re
    import types

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    paths = sorted(glob.glob(os.path.join(root, "profiles", "decode_split_kernel_*.md")))
    assert paths
    for path in paths:
        tag = os.path.basename(path)[len("decode_split_kernel_"):-len(".md")]
        cache = "fp8" if tag.endswith("_fp8") else "bf16"
        name = tag[:-len("_fp8")] if cache == "fp8" else tag
        spec = CONFIGS[name]
        lens = draw_seq_lens(spec["lens"], spec["B"], spec["P"], spec["seed"])
        light = types.SimpleNamespace(B=spec["B"], Hq=spec["Hq"], Hkv=spec["Hkv"], D=spec["D"], P=spec["P"],
                                      seq_lens=torch.from_numpy(lens), qo_indptr=None)
        want = algorithmic_bytes(light, cache=cache)["total"]
        text = open(path).read()
        got = int(re.search(r"algorithmic bytes per launch: ([\d,]+) B", text).group(1).replace(",", ""))
        traffic = int(re.search(r"dram_bytes_per_launch: `(\d+)`", text).group(1))
        assert got == want, (tag, got, want)
        assert want <= traffic <= 1.04 * want, (tag, traffic / want)
        assert re.search(r"kernel_source_hash: `[0-9a-f]{16}`", text), tag
