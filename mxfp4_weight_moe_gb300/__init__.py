"""GB300 (sm_103a) fused MXFP4-weight MoE layer -- placeholder, binding follows."""
