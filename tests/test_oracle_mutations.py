"""The oracles' pins catch planted mistakes.

Each case copies the oracles into a temporary tree, plants one plausible
mistake in the copy and runs that oracle's pins against it: at least one pin
must fail. Decode oracle (pins: tests/test_oracle.py): a wrong head map,
causal offset, LSE base, nibble order, missing scale, sign handling, softmax
scale, slot index, merge weight or scale group. Graph-metadata oracle (pins:
the CPU tests of tests/test_graph_metadata.py): page id from slot, page
position, prefix sums, padding rows. The unmodified copy must pass, so a
failure is the mistake's doing. The oracles in the repository are never
modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (what is planted, text in oracle/decode_ref.py, replacement)
MUTATIONS = [
    ("KV head of query head h taken as h % Hkv", "hk = h // G", "hk = h % Hkv"),
    ("causal offset one key short", "n = L - (Tq - 1) + t", "n = L - Tq + t"),
    ("LSE in log2 instead of ln", "return p @ vals, float(m + math.log(z))",
     "return p @ vals, float(m + math.log2(z))"),
    ("even channel read from the high nibble", "codes[..., 0::2] = lo\n    codes[..., 1::2] = hi",
     "codes[..., 0::2] = hi\n    codes[..., 1::2] = lo"),
    ("INT8 scale dropped", "return codes.astype(np.float64) * scale.astype(np.float64)",
     "return codes.astype(np.float64)"),
    ("INT4 nibbles read unsigned", "return np.where(codes >= 8, codes - 16, codes)", "return codes"),
    ("softmax scale 1/D instead of 1/sqrt(D)", "scale = (1.0 / math.sqrt(D))", "scale = (1.0 / D)"),
    ("slot index off by one", "slots = j % page_size", "slots = (j + 1) % page_size"),
    ("merge weights without the max shift", "w = np.where(np.isfinite(l), np.exp(l - m_safe), 0.0)",
     "w = np.where(np.isfinite(l), np.exp(l), 0.0)"),
    ("INT4 scale groups interleaved", "s = np.repeat(scale.astype(np.float64), 32, axis=-1)[..., :d]",
     "s = np.tile(scale.astype(np.float64), 32)[..., :d]"),
]


# the same for the graph-metadata oracle (oracle/graph_metadata_ref.py), whose
# pins are the CPU tests of tests/test_graph_metadata.py
META_MUTATIONS = [
    ("page id taken from the slot without dividing by P", "page_table[b, j] = slot // P if slot >= 0 else -1",
     "page_table[b, j] = slot if slot >= 0 else -1"),
    ("page j read at position j instead of j * P", "slot = int(req_to_token[r, j * P])",
     "slot = int(req_to_token[r, j])"),
    ("cu_seqlens_k inclusive", "cu_k[b + 1] = cu_k[b] + cache_seqlens[b]",
     "cu_k[b + 1] = cu_k[b] + cache_seqlens[b] + (1 if b == 0 else 0)"),
    ("padding rows keep their query tokens", "cu_q[b + 1] = cu_q[b] + (int(q_in[b]) if idx[b] >= 0 else 0)",
     "cu_q[b + 1] = cu_q[b] + int(q_in[b])"),
]


def _tree(tmp_path):
    """A copy of what the pins need, with the package linked (not copied)."""
    dst = tmp_path / "repo"
    (dst / "tests").mkdir(parents=True)
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), dst / "tests" / "golden")
    for f in ("__init__.py", "conftest.py", "test_oracle.py", "test_graph_metadata.py", "gpu_common.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), dst / "tests" / f)
    os.symlink(os.path.join(ROOT, "split_kv_paged_gqa_gb300"), dst / "split_kv_paged_gqa_gb300")
    return dst


def _run_pins(tree, test_file="tests/test_oracle.py"):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", test_file, "-q", "-x", "-m", "not gpu", "-p",
                        "no:cacheprovider"], cwd=tree, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-400:]


def test_unmodified_copy_passes(tmp_path):
    tree = _tree(tmp_path)
    for f in ("tests/test_oracle.py", "tests/test_graph_metadata.py"):
        code, out = _run_pins(tree, f)
        assert code == 0, out


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, what, old, new):
    tree = _tree(tmp_path)
    src = tree / "oracle" / "decode_ref.py"
    text = src.read_text()
    assert text.count(old) == 1, f"the oracle no longer contains the line this case mutates: {old!r}"
    src.write_text(text.replace(old, new))
    code, out = _run_pins(tree)
    assert code != 0, f"no pin caught: {what}\n{out}"


@pytest.mark.parametrize("what,old,new", META_MUTATIONS, ids=[m[0] for m in META_MUTATIONS])
def test_planted_metadata_mistake_is_caught(tmp_path, what, old, new):
    tree = _tree(tmp_path)
    src = tree / "oracle" / "graph_metadata_ref.py"
    text = src.read_text()
    assert text.count(old) == 1, f"the oracle no longer contains the line this case mutates: {old!r}"
    src.write_text(text.replace(old, new))
    code, out = _run_pins(tree, "tests/test_graph_metadata.py")
    assert code != 0, f"no pin caught: {what}\n{out}"
