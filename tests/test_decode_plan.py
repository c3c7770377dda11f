"""Layer policy of the decode stack, on the host.

"Quest: Query-Aware Sparsity ..." review, section on separating the page count
from the token budget: the first two attention layers keep full attention and
every later layer runs the Quest steps (append, page scores, top-K, attention
over the selected pages). These tests check the routing the stack takes per
layer, without a GPU.
"""
import bench
import workloads
from gqa_head_folding_gb300.decode import layer_plan


def test_first_two_layers_are_dense_then_quest():
    w = workloads.WORKLOADS[3]
    plans = [layer_plan(i, w.k_pages, w.dense_layers, True, True) for i in range(w.num_layers)]
    assert plans[0] == plans[1] == ("append", "dense")
    assert all(p == ("quest",) for p in plans[2:])
    # the fused call appends the token itself; the step-by-step path appends first
    unf = [layer_plan(i, w.k_pages, w.dense_layers, False, True) for i in range(w.num_layers)]
    assert unf[0] == unf[1] == ("append", "dense")
    assert all(p == ("append", "score", "topk", "sparse") for p in unf[2:])


def test_every_layer_appends_when_the_step_carries_a_token():
    for fused in (True, False):
        for i in range(6):
            names = layer_plan(i, 16, 2, fused, True)
            # a Quest layer's metadata is updated on every step, either by the
            # fused call or by an explicit append ahead of the score
            assert "append" in names or "quest" in names


def test_without_a_new_token_no_append_runs():
    assert layer_plan(0, 16, 2, True, False) == ("dense",)
    assert layer_plan(5, 16, 2, False, False) == ("score", "topk", "sparse")
    assert layer_plan(5, 16, 2, True, False) == ("quest",)


def test_dense_only_stacks():
    # no k_pages: every layer dense whatever dense_layers says
    assert all(layer_plan(i, None, 0, True, False) == ("dense",) for i in range(30))
    assert all(layer_plan(i, None, 2, True, True) == ("append", "dense") for i in range(30))


def test_dense_layer_count_is_respected():
    assert [layer_plan(i, 8, 0, True, False) for i in range(3)] == [("quest",)] * 3
    assert [("dense" in layer_plan(i, 8, 3, True, False)) for i in range(5)] == [True] * 3 + [False] * 2


def test_step_bytes_follow_the_same_plan():
    # the bench's per-family launch counts are the plan's call counts
    w = workloads.WORKLOADS[3].with_(num_layers=5)
    lens = [[w.max_len]] * w.num_layers
    for fused in (True, False):
        want = {}
        for i in range(w.num_layers):
            for name in layer_plan(i, w.k_pages, w.dense_layers, fused, w.append):
                want[name] = want.get(name, 0) + 1
        assert bench.step_bytes(w, lens, fused=fused)["launches"] == want
