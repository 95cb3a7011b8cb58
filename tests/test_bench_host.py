"""Host logic of bench.py that needs no GPU: the source digest that ties an ncu summary to the
kernel sources it was captured from, and the traffic figure read back from such a summary."""
import os

import pytest

import bench


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A throw-away repository root with two kernel sources and an empty profiles folder."""
    csrc = tmp_path / "block_diffusion_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_bytes(b"kernel a\n")
    (csrc / "b.cuh").write_bytes(b"header b\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _summary(root, name, digest, traffic):
    (root / "profiles" / f"{name}.md").write_text(
        f"# {name}\n\n- source_sha256: `{digest}` (sha256 of the sources)\n"
        f"- traffic_bytes_per_launch: `{traffic}`\n")


def test_digest_covers_every_source_in_order(tree):
    d = bench.source_digest(("a.cu", "b.cuh"))
    assert d == bench.source_digest(("a.cu", "b.cuh"))
    assert d != bench.source_digest(("b.cuh", "a.cu"))
    (tree / "block_diffusion_gb300" / "csrc" / "b.cuh").write_bytes(b"header b changed\n")
    assert d != bench.source_digest(("a.cu", "b.cuh"))


def test_traffic_only_for_the_sources_it_was_captured_from(tree):
    srcs = ("a.cu", "b.cuh")
    _summary(tree, "k", bench.source_digest(srcs), 123456)
    assert bench.profile_traffic("k", srcs) == 123456.0
    (tree / "block_diffusion_gb300" / "csrc" / "a.cu").write_bytes(b"kernel a, edited\n")
    assert bench.profile_traffic("k", srcs) is None


def test_missing_or_incomplete_summary_gives_no_traffic(tree):
    srcs = ("a.cu",)
    assert bench.profile_traffic("absent", srcs) is None
    (tree / "profiles" / "nodigest.md").write_text("- traffic_bytes_per_launch: `5`\n")
    assert bench.profile_traffic("nodigest", srcs) is None
    (tree / "profiles" / "notraffic.md").write_text(
        f"- source_sha256: `{bench.source_digest(srcs)}`\n")
    assert bench.profile_traffic("notraffic", srcs) is None


def test_committed_summaries_name_real_sources():
    """Every kernel the bench reports has a committed summary and sources that exist."""
    for name, (prof, srcs) in bench.KERNEL_SOURCES.items():
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", f"{prof}.md")), name
        for s in srcs:
            assert os.path.exists(os.path.join(bench.ROOT, "block_diffusion_gb300", "csrc", s)), s
