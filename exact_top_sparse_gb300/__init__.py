"""Sample-guided exact Top-K over ragged FP32 score rows (CUDA, sm_103a)."""
