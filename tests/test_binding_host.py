"""The Python binding's checks, without a GPU.

The C ABI takes plain pointers and sizes, so a buffer shorter than the call
implies cannot be detected there; the binding compares every tensor's shape
with T, V, K and d before any launch.  These tests drive the shape checks with
CPU tensors: the layouts the GPU tests and the benchmark pass are accepted,
and each kind of short or misshapen buffer is refused.  The entry points also
refuse tensors that are not on a CUDA device.
"""

import pytest
import torch

import precision_off_policy_gb300 as sc

T, V, K = 6, 100, 8


def _center(**over):
    a = dict(T=T, V=V, K_max=K,
             logits=torch.empty((T, V), dtype=torch.bfloat16),
             grad_out=torch.empty((T, V), dtype=torch.bfloat16),
             rec_ids=torch.empty((T, K), dtype=torch.int32), rec_logprobs=torch.empty((T, K)),
             rec_count=None, sampled_id=torch.empty(T, dtype=torch.int32), rollout_logprob=torch.empty(T),
             row_response=torch.empty(T, dtype=torch.int32), logp_out=torch.empty(T),
             diag_out=torch.empty((T, 16), dtype=torch.int32), status=torch.empty(1, dtype=torch.int32))
    a.update(over)
    sc._check_center_buffers(a["T"], a["V"], a["K_max"], a["logits"], a["grad_out"], a["rec_ids"],
                             a["rec_logprobs"], a["rec_count"], a["sampled_id"], a["rollout_logprob"],
                             a["row_response"], a["logp_out"], a["diag_out"], a["status"])


def test_center_accepts_the_layouts_in_use():
    _center()
    wide = torch.empty((T, 104), dtype=torch.bfloat16)  # rows padded to a multiple of 8
    _center(logits=wide, grad_out=wide)  # in place, padded stride
    _center(logits=torch.empty((T, 1024), dtype=torch.bfloat16), grad_out=torch.empty((T, 1016), dtype=torch.bfloat16))
    _center(rec_count=torch.empty(T, dtype=torch.int32), rollout_logprob=None, diag_out=None, status=None)
    _center(K_max=0, rec_ids=torch.empty((T, 0), dtype=torch.int32), rec_logprobs=torch.empty((T, 0)))
    _center(K_max=0, rec_ids=None, rec_logprobs=None)
    e = torch.empty((0, K), dtype=torch.int32)
    _center(T=0, logits=torch.empty((0, V), dtype=torch.bfloat16), grad_out=torch.empty((0, V), dtype=torch.bfloat16),
            rec_ids=e, rec_logprobs=e.float(), sampled_id=e[:, 0], rollout_logprob=None, row_response=e[:, 0],
            logp_out=torch.empty(0), diag_out=None)


@pytest.mark.parametrize("over", [
    dict(logits=torch.empty((T, V - 1), dtype=torch.bfloat16)),
    dict(grad_out=torch.empty((T - 1, V), dtype=torch.bfloat16)),
    dict(grad_out=torch.empty((T + 1, V), dtype=torch.bfloat16)),
    dict(grad_out=torch.empty((T, V - 8), dtype=torch.bfloat16)),
    dict(rec_ids=torch.empty((T, K - 1), dtype=torch.int32)),
    dict(rec_logprobs=torch.empty((T - 1, K))),
    dict(rec_ids=None),
    dict(rec_count=torch.empty(T - 1, dtype=torch.int32)),
    dict(sampled_id=torch.empty(T + 1, dtype=torch.int32)),
    dict(rollout_logprob=torch.empty(2)),
    dict(row_response=torch.empty((T, 1), dtype=torch.int32)),
    dict(logp_out=torch.empty(T - 1)),
    dict(diag_out=torch.empty((T, 8), dtype=torch.int32)),
    dict(diag_out=torch.empty((16, T), dtype=torch.int32).t()),
    dict(status=torch.empty(0, dtype=torch.int32)),
])
def test_center_refuses_short_or_misshapen_buffers(over):
    with pytest.raises(ValueError):
        _center(**over)


def _topk(**over):
    a = dict(T=T, V=V, K=K, logits=torch.empty((T, V)), ids_out=torch.empty((T, K), dtype=torch.int32),
             logprobs_out=torch.empty((T, K)), count_out=torch.empty(T, dtype=torch.int32))
    a.update(over)
    sc._check_topk_buffers(a["T"], a["V"], a["K"], a["logits"], a["ids_out"], a["logprobs_out"], a["count_out"])


def test_topk_shapes():
    _topk()
    _topk(logits=torch.empty((T, 104)))  # padded stride, V given
    for over in [dict(logits=torch.empty((T, V - 1))), dict(ids_out=torch.empty((T, K - 1), dtype=torch.int32)),
                 dict(logprobs_out=torch.empty((T - 1, K))), dict(count_out=torch.empty(T + 1, dtype=torch.int32))]:
        with pytest.raises(ValueError):
            _topk(**over)


def _lmhead(**over):
    d = 16
    a = dict(T=T, d=d, V=V, K_max=K, dhidden=torch.empty((T, d), dtype=torch.bfloat16),
             dw=torch.empty((V, d)), rec_ids=torch.empty((T, K), dtype=torch.int32), rec_logprobs=torch.empty((T, K)),
             rec_count=None, sampled_id=torch.empty(T, dtype=torch.int32), rollout_logprob=None,
             row_response=torch.empty(T, dtype=torch.int32), logp_out=torch.empty(T),
             diag_out=torch.empty((T, 16), dtype=torch.int32), status=torch.empty(1, dtype=torch.int32))
    a.update(over)
    sc._check_lmhead_buffers(a["T"], a["d"], a["V"], a["K_max"], a["dhidden"], a["dw"], a["rec_ids"],
                             a["rec_logprobs"], a["rec_count"], a["sampled_id"], a["rollout_logprob"],
                             a["row_response"], a["logp_out"], a["diag_out"], a["status"])


def test_lmhead_shapes():
    _lmhead()
    for over in [dict(dhidden=torch.empty((T, 8), dtype=torch.bfloat16)), dict(dw=torch.empty((V - 1, 16))),
                 dict(dw=torch.empty((16, V)).t()), dict(logp_out=torch.empty(T + 2)),
                 dict(rec_logprobs=torch.empty((T, K + 1)))]:
        with pytest.raises(ValueError):
            _lmhead(**over)


def test_entry_points_refuse_host_tensors():
    r = torch.zeros(8)
    with pytest.raises(ValueError):
        sc.sc_group_advantages(r, 2, 4)
    with pytest.raises(ValueError):
        sc.sc_rollout_mean_advantages(torch.zeros(2), torch.zeros(T, dtype=torch.int32))
    with pytest.raises(ValueError):
        sc.sc_topk_capture(torch.zeros((T, V)), K)
    with pytest.raises(ValueError):
        sc.sc_center_forward_backward(torch.zeros((T, V), dtype=torch.bfloat16), None, None, None,
                                      torch.zeros(T, dtype=torch.int32), None, torch.zeros(T, dtype=torch.int32),
                                      torch.zeros(2), sc.params(K_max=0))
    with pytest.raises(ValueError):
        sc.sc_lmhead_forward_backward(torch.zeros((T, 16), dtype=torch.bfloat16),
                                      torch.zeros((V, 16), dtype=torch.bfloat16), None, None, None,
                                      torch.zeros(T, dtype=torch.int32), None, torch.zeros(T, dtype=torch.int32),
                                      torch.zeros(2), sc.params(K_max=0))
